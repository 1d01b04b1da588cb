// Prefill engine (M > 16 tokens): a dense contraction on the 5th-generation
// tensor cores.
//
// asi.tokyo 2B4T write-up: packed ternary weights are unpacked next to the
// math units and multiplied with 8-bit activations.  B300 (sm_103a) has no
// int8 tcgen05 MMA, so both operands are expanded to f16 in shared memory:
// ternary codes become -1/0/+1 and int8 activations their exact f16 values.
// Every product is an integer of magnitude <= 128 and every partial sum an
// integer below 2^24 for K <= 65536, so the fp32 TMEM accumulator holds
// the exact int32 result.
//
// CTA tile: 128 weight rows (MMA M, TMEM lanes) x BN tokens (MMA N, TMEM
// columns); k advances 64 per pipeline stage (one 128-byte swizzle atom).
// Warps 0-7 are producers: they load packed codes and int8 activations
// (128-bit loads, four stages ahead in registers), expand them and write
// the swizzled K-major tiles, then signal a "full" mbarrier.  One thread of
// warp 8 issues tcgen05.mma (kind::f16, 4 x K16 per stage) and commits to
// the stage's "empty" mbarrier.  After the last stage warps 0-7 read the
// accumulator with tcgen05.ld and apply the rescale epilogue.
// Every mbarrier wait is bounded; an expired wait sets a device status word.
#include "bl_device.cuh"

namespace bl {

__device__ unsigned int g_gemm_status = 0u;

namespace {

constexpr int kStages = 4;
constexpr int kProducers = 256;
constexpr int kThreads = kProducers + 32;
constexpr uint32_t kTileA = 128 * 128;  // 128 rows x 64 f16
constexpr uint32_t kDrainLimit = 1u << 30;

template <int BN>
struct Smem {
    static constexpr uint32_t kTileB = BN * 128;
    static constexpr uint32_t kStage = kTileA + kTileB;
    static constexpr uint32_t kBytes = kStages * kStage + 1024 /*align*/ + 256 /*barriers*/;
};

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const int8_t *__restrict__ q, const float *__restrict__ tok_scale,
                const uint8_t *__restrict__ packed, const float *__restrict__ gamma, int M, int N,
                int K, int KT, int RGN, __nv_bfloat16 *__restrict__ out,
                int32_t *__restrict__ acc_out, uint32_t wait_limit) {
    using L = Smem<BN>;
    constexpr int TPT = kProducers / BN;  // producer threads per token row
    constexpr int NQ = 4 / TPT;           // 16-byte activation chunks per thread per stage
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kStages * L::kStage);
    uint64_t *full = bars, *empty = bars + kStages, *accum = bars + 2 * kStages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * kStages + 1);

    pdl_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int NS = 2 * KT;  // 64-k stages
    bool timed_out = false;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], kProducers);
            mbar_init(&empty[i], 1);
        }
        mbar_init(accum, 1);
        mbar_fence_init();
    }
    if (warp == 8) {
        tmem_alloc(tmem_slot, BN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 8) {
        // ---------------- producers ----------------
        const bool has_a = tid < 128;
        const int rgl = tid >> 4, lc = tid & 15;
        const int ag = lc >> 1, atp = lc & 1;
        const int rg = blockIdx.x * 8 + rgl;
        const int tb = tid / TPT, part = tid % TPT;
        const int tok = blockIdx.y * BN + tb;

        struct Regs {
            uint4 w;
            uint4 x[NQ];
        };
        auto load_w = [&](Regs &r, int st) {
            if (st >= NS) return;
            const int c = st >> 1, hf = st & 1;
            if (has_a && rg < RGN)
                r.w = ld_stream16(packed + (static_cast<int64_t>(rg) * KT + c) * 512 +
                                  16 * (4 * ag + 2 * hf + atp));
            else
                r.w = make_uint4(0x55555555u, 0x55555555u, 0x55555555u, 0x55555555u);
        };
        auto load_x = [&](Regs &r, int st) {
            if (st >= NS) return;
#pragma unroll
            for (int i = 0; i < NQ; ++i) {
                const int k = st * 64 + part * (64 / TPT) + 16 * i;
                r.x[i] = (tok < M && k < K) ? ld_ro16(q + static_cast<int64_t>(tok) * K + k)
                                            : make_uint4(0, 0, 0, 0);
            }
        };
        auto step = [&](const Regs &r, int st) {
            if (st >= NS) return;
            const int slot = st % kStages;
            if (!mbar_wait_bounded(&empty[slot], ((st / kStages) & 1) ^ 1, wait_limit)) timed_out = true;
            uint8_t *sa = smem + slot * L::kStage;
            uint8_t *sb = sa + kTileA;
            if (has_a) {
                const uint32_t wr[4] = {r.w.x, r.w.y, r.w.z, r.w.w};
#pragma unroll
                for (int wi = 0; wi < 4; ++wi) {
                    const int P = wi >> 1, u = wi & 1;
                    const uint32_t row = 16 * rgl + 8 * u + ag;
                    uint32_t f[8];
#pragma unroll
                    for (int p = 0; p < 8; ++p)
                        f[p] = hadd2(((wr[wi] >> (2 * p)) & 0x00030003u) | 0x64006400u,
                                     0xE401E401u);  // (1024 + c) - 1025 = Wq
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t chunk = 4 * atp + 2 * P + h;
                        *reinterpret_cast<uint4 *>(sa + sw128_off(row, chunk)) =
                            make_uint4(f[4 * h], f[4 * h + 1], f[4 * h + 2], f[4 * h + 3]);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < NQ; ++i) {
                const uint32_t xw[4] = {r.x[i].x, r.x[i].y, r.x[i].z, r.x[i].w};
                uint32_t f[8];
#pragma unroll
                for (int wi = 0; wi < 4; ++wi) {
                    const uint32_t x = xw[wi] ^ 0x80808080u;
                    f[2 * wi] = hadd2(prmt(x, 0x64646464u, 0x4140u), 0xE480E480u);  // -1152
                    f[2 * wi + 1] = hadd2(prmt(x, 0x64646464u, 0x4342u), 0xE480E480u);
                }
                const uint32_t chunk = (part * (64 / TPT) + 16 * i) / 8;
                *reinterpret_cast<uint4 *>(sb + sw128_off(tb, chunk)) = make_uint4(f[0], f[1], f[2], f[3]);
                *reinterpret_cast<uint4 *>(sb + sw128_off(tb, chunk + 1)) =
                    make_uint4(f[4], f[5], f[6], f[7]);
            }
            fence_proxy_async_smem();
            mbar_arrive(&full[slot]);
        };

        Regs r0, r1, r2, r3;
        load_w(r0, 0);
        load_w(r1, 1);
        load_w(r2, 2);
        load_w(r3, 3);
        pdl_wait();
        load_x(r0, 0);
        load_x(r1, 1);
        load_x(r2, 2);
        load_x(r3, 3);
        for (int st = 0; st < NS; st += 4) {
            step(r0, st);
            load_w(r0, st + 4);
            load_x(r0, st + 4);
            step(r1, st + 1);
            load_w(r1, st + 5);
            load_x(r1, st + 5);
            step(r2, st + 2);
            load_w(r2, st + 6);
            load_x(r2, st + 6);
            step(r3, st + 3);
            load_w(r3, st + 7);
            load_x(r3, st + 7);
        }
    } else if (lane == 0) {
        // ---------------- MMA issuer ----------------
        constexpr uint32_t idesc = idesc_f16_f32(128, BN);
        const uint32_t base = smem_addr(smem);
        for (int st = 0; st < NS; ++st) {
            const int slot = st % kStages;
            if (!mbar_wait_bounded(&full[slot], (st / kStages) & 1, wait_limit)) timed_out = true;
            tc_fence_after();
            const uint64_t ad = sw128_desc(base + slot * L::kStage);
            const uint64_t bd = sw128_desc(base + slot * L::kStage + kTileA);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                tc_mma_f16(tmem, ad + 2 * kk, bd + 2 * kk, idesc, (st > 0 || kk > 0) ? 1u : 0u);
            tc_commit(&empty[slot]);
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
        // All MMAs must have retired before the accumulator is released.
        if (lane == 0) mbar_wait_bounded(accum, 0, kDrainLimit);
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, BN);
    }
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
    const dim3 grid((RGN + 7) / 8, (M + BN - 1) / BN);
    return launch_pdl(gemm_kernel<BN>, grid, dim3(kThreads), smem, st, 1, q, tok_scale, packed, gamma,
                      M, N, K, KT, RGN, out, acc_out, wait_limit);
}

}  // namespace

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
