// Prefill engine (bitlinear_forward above 64 tokens, bitlinear_forward_f16 at
// any M): a dense contraction on the 5th-generation tensor cores.
//
// asi.tokyo 2B4T write-up, on its GPU kernel (four weights packed per byte):
// packed ternary weights are unpacked next to the math units and multiplied
// with 8-bit activations.  B300 (sm_103a) has no
// int8 tcgen05 MMA, so both operands are fed as f16: ternary codes become
// -1/0/+1 and int8 activations their exact f16 values.  Every product is an
// integer of magnitude <= 128 and every partial sum an integer below 2^24
// for K <= 65536, so the fp32 TMEM accumulator holds the exact int32 result.
//
// CTA tile: 128 weight rows (MMA M, TMEM lanes) x BN tokens (MMA N, TMEM
// columns); k advances 64 per pipeline stage.  Roles:
//   - loader (warp 9, one thread): per stage, a 2-D tensor-map copy of the
//     int8 activation tile (BN tokens x 64 k) and one 3-D tensor-map copy of
//     the eight 512-byte packed weight tiles, into the stage's raw buffers;
//   - converters (warps 0-7): the weight operand A lives in tensor memory:
//     warps 0-3 each own 32 rows (their TMEM lane quarter), expand the
//     row's 2-bit codes to f16 in registers and store them with tcgen05.st;
//     all eight warps expand the int8 tile to f16 into the 128-byte-
//     swizzled K-major B tile in shared memory;
//   - MMA issuer (warp 8, one thread): tcgen05.mma kind::f16, A from TMEM,
//     B from shared memory, 4 x K16 per stage, committed to the stage's
//     "empty" mbarrier.
// No thread waits on a global load in the main loop.  After the last stage
// warps 0-7 read the accumulator with tcgen05.ld and apply the rescale
// epilogue.  Every mbarrier wait is bounded; an expired wait sets a device
// status word.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "bl_device.cuh"

namespace bl {

__device__ unsigned int g_gemm_status = 0u;

namespace {

constexpr int kRaw = 6;    // raw (packed weights + int8 activations) stages in flight
constexpr int kOps = 3;    // operand stages (f16 activation tile + weight TMEM columns)
constexpr int kConverters = 256;                // warps 0-7
constexpr int kThreads = kConverters + 64;      // + MMA warp 8 + loader warp 9
constexpr uint32_t kDrainLimit = 1u << 30;
constexpr uint32_t kRawA = 8 * 512;             // packed codes of 8 row groups, one k-tile

template <int BN>
struct Smem {
    static constexpr uint32_t kTileB = BN * 128;        // f16 tile, BN tokens x 64 k, swizzled
    static constexpr uint32_t kRawB = BN * 64;              // int8 tile, BN tokens x 64 k
    static constexpr uint32_t kRawStage = kRawA + kRawB;    // packed codes | int8 tile
    static constexpr uint32_t kRawBase = kOps * kTileB;     // operand tiles first: 1024-aligned
    static constexpr uint32_t kBytes = kRawBase + kRaw * kRawStage + 1024 /*align*/ + 256 /*barriers*/;
    // TMEM: accumulator in columns [0, BN), weight stages after it (32 columns each)
    static constexpr uint32_t kACol = BN;
    static constexpr uint32_t kCols = BN + 32 * kOps <= 256 ? 256 : 512;
};

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// Packed weights of 8 row groups at one 128-k tile, by one tensor-map copy:
// the packed buffer seen as u64 [row group][k-tile][64], box 64 x 1 x 8
// (4 KB, row group major, so the 512-byte tiles land back to back).  One
// copy instead of eight 512-byte bulk copies: the copy instructions, issued
// by one loader thread, set the pace of the pipeline.
__device__ __forceinline__ void tma_load_w8(void *dst, const CUtensorMap *map, int c, int rg0, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(c), "r"(rg0), "r"(smem_addr(bar))
        : "memory");
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap wmap,
                const float *__restrict__ tok_scale,
                const uint8_t *__restrict__ packed, const float *__restrict__ gamma, int M, int N,
                int K, int KT, int RGN, __nv_bfloat16 *__restrict__ out,
                int32_t *__restrict__ acc_out, uint32_t wait_limit) {
    using L = Smem<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kRawBase + kRaw * L::kRawStage);
    uint64_t *raw_full = bars, *raw_empty = bars + kRaw;
    uint64_t *mma_full = bars + 2 * kRaw, *op_empty = bars + 2 * kRaw + kOps;
    uint64_t *accum = bars + 2 * kRaw + 2 * kOps;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(accum + 1);
    int *issued = reinterpret_cast<int *>(tmem_slot + 1);  // stages whose copies the loader issued

    pdl_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int NS = 2 * KT;  // 64-k stages
    bool timed_out = false;

    if (tid == 0) {
        *issued = 0;
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
        tmem_alloc(tmem_slot, L::kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int rg0 = blockIdx.x * 8;
    const int nrg = RGN - rg0 < 8 ? RGN - rg0 : 8;

    if (warp == 9) {
        // ---------------- loader ----------------
        if (lane == 0) {
            const uint32_t bytes = kRawA + L::kRawB;  // a full box: rows past N arrive zero-filled (unread)
            // the packed weights are static: their copies may start before the
            // previous kernel finished; the activations may not
            bool waited = false;
            for (int st = 0; st < NS; ++st) {
                const int rs = st % kRaw;
                if (!mbar_wait_bounded(&raw_empty[rs], ((st / kRaw) & 1) ^ 1, wait_limit)) {
                    timed_out = true;
                    break;
                }
                uint8_t *raw = smem + L::kRawBase + rs * L::kRawStage;
                mbar_arrive_expect_tx(&raw_full[rs], bytes);
                tma_load_w8(raw, &wmap, st >> 1, rg0, &raw_full[rs]);
                if (!waited) {
                    pdl_wait();
                    waited = true;
                }
                tma_load_2d(raw + kRawA, &qmap, st * 64, blockIdx.y * BN, &raw_full[rs]);
                *issued = st + 1;
            }
        }
    } else if (warp < 8) {
        // Warp w owns TMEM lane quarter w % 4 (weight rows 32(w%4) + lane)
        // and half t' = w / 4 of each stage's 32 weight columns.
        const int row = 32 * (warp & 3) + lane;
        const int ri = row & 15, rgl = row >> 4, t2 = warp >> 2;
        const bool row_ok = rgl < nrg;
        const uint32_t a_off = 512 * rgl + 16 * 4 * (ri & 7) + 4 * (ri >> 3);
        const uint32_t a_lane = static_cast<uint32_t>(32 * (warp & 3)) << 16;
        for (int st = 0; st < NS; ++st) {
            const int rs = st % kRaw, slot = st % kOps;
            if (!mbar_wait_bounded(&raw_full[rs], (st / kRaw) & 1, wait_limit)) timed_out = true;
            if (!mbar_wait_bounded(&op_empty[slot], ((st / kOps) & 1) ^ 1, wait_limit)) timed_out = true;
            const uint8_t *raw = smem + L::kRawBase + rs * L::kRawStage;
            uint8_t *stage = smem + slot * L::kTileB;
            {
                // column c of the stage holds k = 2c, 2c+1: word (t' = c/16, P = (c%16)/8), pair p = c%8
                const int hf = st & 1;
                uint32_t f[16];
#pragma unroll
                for (int P = 0; P < 2; ++P) {
                    const uint32_t w = row_ok ? *reinterpret_cast<const uint32_t *>(
                                                    raw + a_off + 16 * (2 * hf + t2) + 8 * P)
                                              : 0x55555555u;
#pragma unroll
                    for (int p = 0; p < 8; ++p)
                        f[8 * P + p] = hadd2(((w >> (2 * p)) & 0x00030003u) | 0x64006400u, 0xE401E401u);  // Wq
                }
                tc_st16(tmem + a_lane + L::kACol + 32 * slot + 16 * t2, f);
            }
            // int8 tile (token-major, 64 bytes per token) -> swizzled f16 tile
            const uint8_t *rb = raw + kRawA;
#pragma unroll
            for (int j = 0; j < BN * 4 / kConverters; ++j) {
                const int e = tid + kConverters * j;
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
    } else if (lane == 0) {
        // ---------------- MMA issuer ----------------
        constexpr uint32_t idesc = idesc_f16_f32(128, BN);
        const uint32_t base = smem_addr(smem);
        for (int st = 0; st < NS; ++st) {
            const int slot = st % kOps;
            if (!mbar_wait_bounded(&mma_full[slot], (st / kOps) & 1, wait_limit)) timed_out = true;
            tc_fence_after();
            const uint64_t bd = sw128_desc(base + slot * L::kTileB);
            const uint32_t at = tmem + L::kACol + 32 * slot;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                tc_mma_f16_ta(tmem, at + 8 * kk, bd + 2 * kk, idesc, (st > 0 || kk > 0) ? 1u : 0u);
            tc_commit(&op_empty[slot]);
        }
        tc_commit(accum);
    }

    // ---------------- epilogue (warps 0-7) ----------------
    if (warp < 8) {
        if (!mbar_wait_bounded(accum, 0, wait_limit)) timed_out = true;
        tc_fence_after();
        const int lq = warp & 3, ch = warp >> 2;
        const float gam = *gamma;
        const int n = blockIdx.x * 128 + 32 * lq + lane;
#pragma unroll 1
        for (int col = ch * (BN / 2); col < (ch + 1) * (BN / 2); col += 16) {
            uint32_t v[16];
            tc_ld16(tmem + (static_cast<uint32_t>(32 * lq) << 16) + col, v);
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int tk = blockIdx.y * BN + col + i;
                if (tk < M && n < N) {
                    const int a = __float2int_rn(__uint_as_float(v[i]));
                    const float f = __fmul_rn(gam, tok_scale[tk]);
                    out[static_cast<int64_t>(tk) * N + n] =
                        __float2bfloat16_rn(__fmul_rn(static_cast<float>(a), f));
                    if (acc_out) acc_out[static_cast<int64_t>(tk) * N + n] = a;
                }
            }
        }
    }
    if (timed_out) atomicOr(&g_gemm_status, 1u);
    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        // All MMAs must have retired, and every copy landed, before the
        // accumulator and shared memory are released.
        if (lane == 0) {
            mbar_wait_bounded(accum, 0, kDrainLimit);
            const int n = *issued;  // only copies that were issued can be in flight
            for (int st = n > kRaw ? n - kRaw : 0; st < n; ++st)
                mbar_wait_bounded(&raw_full[st % kRaw], (st / kRaw) & 1, kDrainLimit);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, L::kCols);
    }
}

// ---------------------------------------------------------------------------
// Variant with f16 activations (bitlinear_quant_act_f16): the activation
// tile arrives by tensor-map copy already in the 128-byte-swizzled K-major
// layout the MMA reads, so the converter warps only expand the weight codes
// into tensor memory.  Stage = swizzled f16 tile | packed codes.
// ---------------------------------------------------------------------------
// NSTG stages; MINB CTAs per SM (a template parameter: with 2, one CTA's
// prologue and epilogue could run under the other's main loop, but the
// TMEM columns of both must then fit in 512; every launch uses MINB = 1).
template <int BN, int NSTG>
struct Smem16 {
    static constexpr uint32_t kTileB = BN * 128;
    static constexpr uint32_t kStage = kTileB + kRawA;  // multiple of 1024
    static constexpr uint32_t kBytes = NSTG * kStage + 1024 /*align*/ + 256 /*barriers*/;
    static constexpr uint32_t kACol = BN;
    static constexpr uint32_t kCols = BN + 32 * NSTG <= 128 ? 128 : (BN + 32 * NSTG <= 256 ? 256 : 512);
};

template <int BN, int NSTG, int MINB>
__global__ void __launch_bounds__(kThreads, MINB)
    gemm16_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap wmap,
                  const float *__restrict__ tok_scale,
                  const uint8_t *__restrict__ packed, const float *__restrict__ gamma, int M, int N,
                  int K, int KT, int RGN, __nv_bfloat16 *__restrict__ out,
                  int32_t *__restrict__ acc_out, uint32_t wait_limit) {
    using L = Smem16<BN, NSTG>;
    static_assert(MINB * L::kCols <= 512, "the CTAs of an SM share 512 TMEM columns");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + NSTG * L::kStage);
    uint64_t *full = bars, *a_ready = bars + NSTG, *empty = bars + 2 * NSTG;
    uint64_t *accum = bars + 3 * NSTG;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(accum + 1);
    int *issued = reinterpret_cast<int *>(tmem_slot + 1);

    pdl_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int NS = 2 * KT;  // 64-k stages
    bool timed_out = false;
    if (tid == 0) {
        *issued = 0;
        for (int i = 0; i < NSTG; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&a_ready[i], kConverters / 2);
            mbar_init(&empty[i], 1);
        }
        mbar_init(accum, 1);
        mbar_fence_init();
    }
    if (warp == 8) {
        tmem_alloc(tmem_slot, L::kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int rg0 = blockIdx.x * 8;
    const int nrg = RGN - rg0 < 8 ? RGN - rg0 : 8;

    if (warp == 9) {
        // ---------------- loader ----------------
        if (lane == 0) {
            const uint32_t bytes = kRawA + L::kTileB;  // a full box: rows past N arrive zero-filled (unread)
            bool waited = false;
            for (int st = 0; st < NS; ++st) {
                const int s = st % NSTG;
                if (!mbar_wait_bounded(&empty[s], ((st / NSTG) & 1) ^ 1, wait_limit)) {
                    timed_out = true;
                    break;
                }
                uint8_t *stage = smem + s * L::kStage;
                mbar_arrive_expect_tx(&full[s], bytes);
                tma_load_w8(stage + L::kTileB, &wmap, st >> 1, rg0, &full[s]);
                if (!waited) {  // the weights are static; the activations come from earlier kernels
                    pdl_wait();
                    waited = true;
                }
                tma_load_2d(stage, &qmap, st * 64, blockIdx.y * BN, &full[s]);
                *issued = st + 1;
            }
        }
    } else if (warp < 8) {
        // ---------------- converters: weight codes -> f16 in TMEM ----------------
        // Warp w owns TMEM lane quarter w % 4 (weight rows 32(w%4) + lane) and
        // the stages of parity w / 4, so two stages are converted at once.
        const int row = 32 * (warp & 3) + lane;
        const int ri = row & 15, rgl = row >> 4;
        const bool row_ok = rgl < nrg;
        const uint32_t a_off = 512 * rgl + 16 * 4 * (ri & 7) + 4 * (ri >> 3);
        const uint32_t a_lane = static_cast<uint32_t>(32 * (warp & 3)) << 16;
        for (int st = warp >> 2; st < NS; st += 2) {
            const int s = st % NSTG;
            if (!mbar_wait_bounded(&full[s], (st / NSTG) & 1, wait_limit)) timed_out = true;
            const uint8_t *codes = smem + s * L::kStage + L::kTileB;
            const int hf = st & 1;
#pragma unroll
            for (int t2 = 0; t2 < 2; ++t2) {  // two 16-column halves (fewer live registers)
                uint32_t f[16];
#pragma unroll
                for (int P = 0; P < 2; ++P) {
                    const uint32_t w = row_ok ? *reinterpret_cast<const uint32_t *>(codes + a_off + 16 * (2 * hf + t2) + 8 * P)
                                              : 0x55555555u;
#pragma unroll
                    for (int p = 0; p < 8; ++p)
                        f[8 * P + p] = hadd2(((w >> (2 * p)) & 0x00030003u) | 0x64006400u, 0xE401E401u);
                }
                tc_st16(tmem + a_lane + L::kACol + 32 * s + 16 * t2, f);
            }
            tc_wait_st();
            tc_fence_before();
            mbar_arrive(&a_ready[s]);
        }
    } else if (lane == 0) {
        // ---------------- MMA issuer ----------------
        constexpr uint32_t idesc = idesc_f16_f32(128, BN);
        const uint32_t base = smem_addr(smem);
        for (int st = 0; st < NS; ++st) {
            const int s = st % NSTG;
            if (!mbar_wait_bounded(&full[s], (st / NSTG) & 1, wait_limit)) timed_out = true;
            if (!mbar_wait_bounded(&a_ready[s], (st / NSTG) & 1, wait_limit)) timed_out = true;
            tc_fence_after();
            const uint64_t bd = sw128_desc(base + s * L::kStage);
            const uint32_t at = tmem + L::kACol + 32 * s;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                tc_mma_f16_ta(tmem, at + 8 * kk, bd + 2 * kk, idesc, (st > 0 || kk > 0) ? 1u : 0u);
            tc_commit(&empty[s]);
        }
        tc_commit(accum);
    }

    // ---------------- epilogue (warps 0-7) ----------------
    if (warp < 8) {
        if (!mbar_wait_bounded(accum, 0, wait_limit)) timed_out = true;
        tc_fence_after();
        const int lq = warp & 3, ch = warp >> 2;
        const float gam = *gamma;
        const int n = blockIdx.x * 128 + 32 * lq + lane;
#pragma unroll 1
        for (int col = ch * (BN / 2); col < (ch + 1) * (BN / 2); col += 16) {
            uint32_t v[16];
            tc_ld16(tmem + (static_cast<uint32_t>(32 * lq) << 16) + col, v);
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int tk = blockIdx.y * BN + col + i;
                if (tk < M && n < N) {
                    const int a = __float2int_rn(__uint_as_float(v[i]));
                    const float f = __fmul_rn(gam, tok_scale[tk]);
                    out[static_cast<int64_t>(tk) * N + n] =
                        __float2bfloat16_rn(__fmul_rn(static_cast<float>(a), f));
                    if (acc_out) acc_out[static_cast<int64_t>(tk) * N + n] = a;
                }
            }
        }
    }
    if (timed_out) atomicOr(&g_gemm_status, 1u);
    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        if (lane == 0) {
            mbar_wait_bounded(accum, 0, kDrainLimit);
            const int n = *issued;  // only copies that were issued can be in flight
            for (int st = n > NSTG ? n - NSTG : 0; st < n; ++st)
                mbar_wait_bounded(&full[st % NSTG], (st / NSTG) & 1, kDrainLimit);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, L::kCols);
    }
}

// Tensor map of the int8 activations [M, K] (row-major): BN x 64 boxes.
std::mutex g_encode_mutex;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// The driver's tensor-map encoder, looked up once.
cudaError_t tensor_map_encoder() {
    std::lock_guard<std::mutex> lock(g_encode_mutex);
    if (!g_encode) {
        cudaDriverEntryPointQueryResult qr;
        void *fn = nullptr;
        cudaError_t e = cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &fn, cudaEnableDefault, &qr);
        if (e != cudaSuccess || qr != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    return cudaSuccess;
}

cudaError_t make_qmap(CUtensorMap *map, const void *q, int M, int K, int BN, bool f16) {
    cudaError_t e0 = tensor_map_encoder();
    if (e0 != cudaSuccess) return e0;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * (f16 ? 2u : 1u)};
    const cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(BN)};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = g_encode(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                                const_cast<void *>(q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                f16 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Tensor map of the packed weights (layout of bitlinear_packed_bytes): u64
// [RGN][KT][64], boxes of 64 x 1 x 8.
cudaError_t make_wmap(CUtensorMap *map, const uint8_t *packed, int RGN, int KT) {
    cudaError_t e = tensor_map_encoder();
    if (e != cudaSuccess) return e;
    const cuuint64_t dims[3] = {64u, static_cast<cuuint64_t>(KT), static_cast<cuuint64_t>(RGN)};
    const cuuint64_t strides[2] = {512u, static_cast<cuuint64_t>(KT) * 512u};
    const cuuint32_t box[3] = {64u, 1u, 8u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<uint8_t *>(packed), dims, strides,
                                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int BN, int NSTG, int MINB>
cudaError_t launch16_bn(const void *q16, const float *tok_scale, const uint8_t *packed, const float *gamma,
                        int M, int N, int K, __nv_bfloat16 *out, int32_t *acc_out, cudaStream_t st,
                        uint32_t wait_limit) {
    const int KT = (K + 127) / 128;
    const int RGN = (N + 15) / 16;
    const uint32_t smem = Smem16<BN, NSTG>::kBytes;
    static bool configured[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(gemm16_kernel<BN, NSTG, MINB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    CUtensorMap qmap, wmap;
    e = make_qmap(&qmap, q16, M, K, BN, true);
    if (e != cudaSuccess) return e;
    e = make_wmap(&wmap, packed, RGN, KT);
    if (e != cudaSuccess) return e;
    const dim3 grid((RGN + 7) / 8, (M + BN - 1) / BN);
    return launch_pdl(gemm16_kernel<BN, NSTG, MINB>, grid, dim3(kThreads), smem, st, 1, qmap, wmap, tok_scale, packed, gamma,
                      M, N, K, KT, RGN, out, acc_out, wait_limit);
}

template <int BN>
cudaError_t launch_bn(const int8_t *q, const float *tok_scale, const uint8_t *packed,
                      const float *gamma, int M, int N, int K, __nv_bfloat16 *out,
                      int32_t *acc_out, cudaStream_t st, uint32_t wait_limit) {
    const int KT = (K + 127) / 128;
    const int RGN = (N + 15) / 16;
    const uint32_t smem = Smem<BN>::kBytes;
    static bool configured[64] = {false};  // the attribute is set once per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(gemm_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    CUtensorMap qmap, wmap;
    e = make_qmap(&qmap, q, M, K, BN, false);
    if (e != cudaSuccess) return e;
    e = make_wmap(&wmap, packed, RGN, KT);
    if (e != cudaSuccess) return e;
    const dim3 grid((RGN + 7) / 8, (M + BN - 1) / BN);
    return launch_pdl(gemm_kernel<BN>, grid, dim3(kThreads), smem, st, 1, qmap, wmap, tok_scale, packed, gamma,
                      M, N, K, KT, RGN, out, acc_out, wait_limit);
}

}  // namespace

// Token tile (MMA N) of the f16 GEMM for M > 128, one CTA per SM holding a
// 128-row x BN tile: 256, or 192 where that takes fewer whole waves.  A 64-k
// stage costs about the same down to BN = 192 (its copies and weight
// conversion set a floor), so a narrower tile pays only where the wave count
// drops: e.g. N = 2560 (20 row tiles) at M = 4096 gives 320 tiles with
// BN = 256 (2.2 waves, three paid) and 440 with BN = 192 (three full waves).
int token_tile(int M, int N) {
    int sms = 148, dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t row_tiles = (N + 127) / 128;
    auto cost = [&](int bn) {  // whole waves x a per-tile time with a large fixed part
        const int64_t tiles = row_tiles * ((M + bn - 1) / bn);
        return (tiles + sms - 1) / sms * (bn + 64);
    };
    return cost(192) < cost(256) ? 192 : 256;
}

cudaError_t launch_gemm16(const void *q16, const float *tok_scale, const uint8_t *packed,
                          const float *gamma, int M, int N, int K, __nv_bfloat16 *out,
                          int32_t *acc_out, cudaStream_t st, uint32_t wait_limit) {
    if (M <= 64) return launch16_bn<64, 6, 1>(q16, tok_scale, packed, gamma, M, N, K, out, acc_out, st, wait_limit);
    if (M <= 128) return launch16_bn<128, 6, 1>(q16, tok_scale, packed, gamma, M, N, K, out, acc_out, st, wait_limit);
    if (token_tile(M, N) == 192)
        return launch16_bn<192, 6, 1>(q16, tok_scale, packed, gamma, M, N, K, out, acc_out, st, wait_limit);
    return launch16_bn<256, 6, 1>(q16, tok_scale, packed, gamma, M, N, K, out, acc_out, st, wait_limit);
}

cudaError_t launch_gemm(const int8_t *q, const float *tok_scale, const uint8_t *packed,
                        const float *gamma, int M, int N, int K, __nv_bfloat16 *out,
                        int32_t *acc_out, cudaStream_t st, uint32_t wait_limit) {
    if (M <= 64) return launch_bn<64>(q, tok_scale, packed, gamma, M, N, K, out, acc_out, st, wait_limit);
    if (M <= 128) return launch_bn<128>(q, tok_scale, packed, gamma, M, N, K, out, acc_out, st, wait_limit);
    return launch_bn<256>(q, tok_scale, packed, gamma, M, N, K, out, acc_out, st, wait_limit);
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
