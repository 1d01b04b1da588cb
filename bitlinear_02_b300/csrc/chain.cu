// Fused decode chain (M <= 16 tokens): a sequence of BitLinear projections,
// each quantising its input (RMSNorm + per-token absmax int8) and multiplying
// it with ternary weights, run as ONE persistent kernel.
//
// The BitLinear layer (cheatsheet.md, "BitNet b1.58とは？"; asi.tokyo 2B4T
// write-up) quantises every projection's input per token from its absolute
// maximum, so a projection cannot start before the whole output vector of
// the projection feeding it is known.  In a decode step those global
// dependencies, not the weight bytes, set the time: a 2560x2560 layer is
// 1.6 MB of packed weights, 0.25 us at HBM speed, while a kernel boundary or
// a grid barrier costs about 1 us.  This engine therefore:
//   - keeps one CTA per SM resident for the whole chain;
//   - streams every CTA's packed weights for ALL projections, in the order it
//     will use them, into a shared-memory ring with bulk async copies (one
//     producer warp), so HBM keeps streaming while the CTAs wait on
//     dependencies;
//   - fuses the quantiser: each projection's epilogue publishes, per CTA,
//     the max |v| and sum v^2 of the outputs it finished; the consumers of
//     that output combine the partials (in a fixed order) into the token's
//     absmax scale and RMS factor, and quantise their slice of the input
//     while loading it;
//   - synchronises phases with a relaxed arrival counter (no memory fences)
//     and makes every exchanged word self-validating: each 64-bit word
//     carries a tag (launch epoch, phase) next to its payload, and a reader
//     re-reads until the tag matches.
// Work split of a phase (projections sharing one input): the CTAs form G
// groups of S; a group owns a contiguous range of 16-row groups, and CTA s
// of the group multiplies K-slice s of them.  Partial sums of a K-split are
// exchanged as tagged words and each CTA finishes a share of the group's
// rows.  The MMA arithmetic is the decode GEMV's (decode_math.cuh): exact
// int32 accumulators, identical results to bitlinear_quant_act followed by
// bitlinear_forward, up to the token scale's last bits (a float reduction).
#include <cstring>
#include <mutex>
#include <vector>

#include "decode_math.cuh"

namespace bl {
cudaError_t status_word(unsigned int **dev_ptr);  // gemm.cu: the library's device status word

namespace chain {

constexpr int kConsumerWarps = 7;  // + 1 producer warp: 8 warps, so 255 registers fit
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kThreads = kConsumers + 32;
constexpr int kDesc = 32;          // weight chunks in flight per CTA (one per task)
constexpr int kMaxProjPerPhase = 4;
constexpr int kMaxProj = 1024;     // gamma values staged in shared memory
constexpr int kMaxCTA = 256;
constexpr uint32_t kDrainLimit = 1u << 30;
constexpr uint64_t kPlanMagic = 0x424c4348414e3031ull;

struct Proj {
    const uint8_t *packed;
    const float *gamma;
    __nv_bfloat16 *out;
    int32_t *acc_out;
    float *tok_scale_out;
    unsigned long long *act_out;    // tagged outputs [M][N/2] if a later projection reads them
    unsigned long long *stats_out;  // tagged per-CTA statistics [nCTA][Mp] if read later
    int32_t N, RG, rg_base, pad;
};

struct Phase {
    const unsigned long long *act_in;    // tagged input, or NULL for the chain input x
    const unsigned long long *stats_in;  // tagged statistics of the input
    int32_t K, KT, S, G;
    int32_t proj0, nproj, RGT, in_phase;  // in_phase: phase index that wrote the input
    int32_t qstride, rg_max, pad0, pad1;
};
static_assert(sizeof(Phase) % 16 == 0 && sizeof(Proj) % 8 == 0, "plan records");

// Metadata image of one phase (contiguous, so one round trip fetches it).
struct MetaImg {
    Phase ph;
    Proj pj[kMaxProjPerPhase];
};

struct Args {
    const MetaImg *metas;
    const float *const *gammas;  // device pointers of every projection's gamma
    const __nv_bfloat16 *x;
    unsigned long long *x_stats;
    unsigned long long *partials;
    unsigned int *ctl;     // [0] arrivals, [1] exits, [2] launch epoch
    unsigned int *status;  // library status word (bounded wait expired)
    int32_t nphase, nproj, M, Mp, nCTA, K0;
    uint32_t ring_bytes, q_bytes, part_bytes, wait_limit;
    float eps;
};

// ------------------------------------------------------------ work split --

struct Work {
    int g, s, r0, r1, t0, t1, nrgs, nsets, npieces;
    bool valid;
};

__host__ __device__ inline Work work_of(const Phase &ph, int cta) {
    Work w{};
    w.s = cta % ph.S;
    w.g = cta / ph.S;
    w.valid = w.g < ph.G;
    if (!w.valid) return w;
    w.r0 = static_cast<int>(static_cast<int64_t>(w.g) * ph.RGT / ph.G);
    w.r1 = static_cast<int>(static_cast<int64_t>(w.g + 1) * ph.RGT / ph.G);
    w.t0 = w.s * ph.KT / ph.S;
    w.t1 = (w.s + 1) * ph.KT / ph.S;
    w.nrgs = w.r1 - w.r0;
    w.nsets = (w.nrgs + 3) / 4;
    const int kt = w.t1 - w.t0;
    if (w.nsets == 0 || kt <= 0) {
        w.npieces = 0;
        return w;
    }
    const int by_size = (kt + 7) / 8;
    const int by_warps = (kConsumerWarps + w.nsets - 1) / w.nsets;
    const int pieces = by_warps < kt ? by_warps : kt;
    w.npieces = by_size > pieces ? by_size : pieces;
    return w;
}

// Task i of a CTA's phase work: up to 4 row groups x up to 8 k-tiles; its
// weights travel as one chunk of the shared-memory ring.
struct Task {
    int rlo, rhi, tlo, thi;
};

__host__ __device__ inline Task task_of(const Work &w, int i) {
    Task t;
    const int set = i / w.npieces, piece = i % w.npieces;
    t.rlo = w.r0 + 4 * set;
    t.rhi = t.rlo + 4 < w.r1 ? t.rlo + 4 : w.r1;
    const int kt = w.t1 - w.t0;
    t.tlo = w.t0 + piece * kt / w.npieces;
    t.thi = w.t0 + (piece + 1) * kt / w.npieces;
    return t;
}

constexpr int kMetaWords = static_cast<int>(sizeof(MetaImg) / 4);
constexpr int kMetaPerLane = (kMetaWords + 31) / 32;

// Shared-memory layout (bytes): ring | q cache | partial sums | metadata x2 |
// mbarriers | chunk offsets | reductions | scalars.
__host__ __device__ inline uint32_t smem_fixed_bytes() {
    return 2 * static_cast<uint32_t>(sizeof(MetaImg)) + kMaxProj * 4 + 2 * kDesc * 8 + kDesc * 4 +
           kConsumerWarps * kMaxProjPerPhase * 16 * 12 + 16 * 4 * 2 + 64;
}
__host__ __device__ inline uint32_t smem_bytes_for(uint32_t ring, uint32_t q_bytes, uint32_t part_bytes) {
    return ring + q_bytes + part_bytes + smem_fixed_bytes();
}

// ------------------------------------------------------------- device ----

// Tags: 32-bit (launch epoch, phase index); the launch epoch starts at 1, so
// a cleared word (tag 0) never matches.  Statistics words carry a 16-bit
// tag, mapped to 1..65535 for the same reason.
__device__ __forceinline__ uint32_t tag_of(uint32_t epoch, int phase_idx) {
    return epoch * 1024u + static_cast<uint32_t>(phase_idx);
}
__device__ __forceinline__ uint32_t tag16_of(uint32_t tag) { return tag % 65535u + 1u; }

struct Shared {
    uint8_t *ring, *qc;
    int32_t *part;
    MetaImg *meta;    // [2]
    float *gall;      // gamma of every projection
    uint64_t *full, *empty;
    uint32_t *coff;   // ring offset (monotonic) of each chunk descriptor
    float *red_hi, *red_lo;  // [warp][proj][16]
    float *red_mx;           // [warp][proj][16]
    float *c, *ts;
    volatile int *abort_flag;
    uint32_t *epoch;
};

__device__ __forceinline__ Shared carve(uint8_t *base, const Args &A) {
    Shared S;
    S.ring = base;
    S.qc = base + A.ring_bytes;
    S.part = reinterpret_cast<int32_t *>(S.qc + A.q_bytes);
    uint8_t *p = reinterpret_cast<uint8_t *>(S.part) + A.part_bytes;
    S.meta = reinterpret_cast<MetaImg *>(p);
    p += 2 * sizeof(MetaImg);
    S.gall = reinterpret_cast<float *>(p);
    p += kMaxProj * 4;
    S.full = reinterpret_cast<uint64_t *>(p);
    S.empty = S.full + kDesc;
    S.coff = reinterpret_cast<uint32_t *>(S.empty + kDesc);
    S.red_hi = reinterpret_cast<float *>(S.coff + kDesc);
    S.red_lo = S.red_hi + kConsumerWarps * kMaxProjPerPhase * 16;
    S.red_mx = S.red_lo + kConsumerWarps * kMaxProjPerPhase * 16;
    S.c = S.red_mx + kConsumerWarps * kMaxProjPerPhase * 16;
    S.ts = S.c + 16;
    S.abort_flag = reinterpret_cast<volatile int *>(S.ts + 16);
    S.epoch = reinterpret_cast<uint32_t *>(S.ts + 16) + 1;
    return S;
}

__device__ __forceinline__ void raise_abort(const Shared &S, unsigned int *status) {
    *S.abort_flag = 1;
    atomicOr(status, 1u);
}

// Re-read a tagged word until (word >> shift) & mask == want, backing off
// between reads.  Returns the word; on timeout, or when another CTA
// reported a failure, returns it with the tag field cleared (never a valid
// tag), which the caller treats as failure.  Out of line: the slow path.
__device__ __noinline__ unsigned long long poll_tag(const unsigned long long *p, uint32_t want, uint32_t mask,
                                                    int shift, uint32_t limit, const unsigned *status) {
    for (uint32_t i = 0; i < limit; ++i) {
        __nanosleep(32);
        const unsigned long long v = ld_cg_u64(p);
        if (static_cast<uint32_t>(v >> shift & mask) == want) return v;
        if ((i & 63u) == 63u && (ld_relaxed_u32(status) & 1u) != 0u) break;  // another CTA gave up
    }
    return 0ull;
}
__device__ __forceinline__ bool tag_ok(unsigned long long v, uint32_t want, uint32_t mask, int shift) {
    return static_cast<uint32_t>(v >> shift & mask) == want;
}

// Compensated fp32 sums (hi + lo, error-free two-sum steps): B300's FP64
// units are far too slow for this path.  Squares of bf16 values are exact in
// fp32, so a sum of squares carries about 2^-48 relative error.
struct FF {
    float hi = 0.0f, lo = 0.0f;
    __device__ __forceinline__ void add(float p) {
        const float s = __fadd_rn(hi, p);
        const float bp = __fsub_rn(s, hi);
        lo = __fadd_rn(lo, __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(p, bp)));
        hi = s;
    }
    __device__ __forceinline__ void add(const FF &o) {
        add(o.hi);
        lo = __fadd_rn(lo, o.lo);
    }
    __device__ __forceinline__ void add_sq(float v) { add(__fmul_rn(v, v)); }
    __device__ __forceinline__ float value() const { return __fadd_rn(hi, lo); }
};

// Per-token reduction of (max, sum of squares) over the consumer
// threads, where thread t holds token t % Mp: a fixed shuffle tree, then a
// fixed-order sum over warps (combine_stats).
__device__ __forceinline__ void reduce_stats(const Shared &S, int j, float mx, FF ss, int Mp, int warp,
                                             int lane) {
    for (int off = 16; off >= Mp; off >>= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        FF o;
        o.hi = __shfl_xor_sync(0xffffffffu, ss.hi, off);
        o.lo = __shfl_xor_sync(0xffffffffu, ss.lo, off);
        ss.add(o);
    }
    if (lane < Mp) {
        S.red_mx[(warp * kMaxProjPerPhase + j) * 16 + lane] = mx;
        S.red_hi[(warp * kMaxProjPerPhase + j) * 16 + lane] = ss.hi;
        S.red_lo[(warp * kMaxProjPerPhase + j) * 16 + lane] = ss.lo;
    }
}
__device__ __forceinline__ void combine_stats(const Shared &S, int j, int m, float &mx, FF &ss) {
    mx = 0.0f;
    ss = FF();
    for (int w = 0; w < kConsumerWarps; ++w) {
        mx = fmaxf(mx, S.red_mx[(w * kMaxProjPerPhase + j) * 16 + m]);
        FF o;
        o.hi = S.red_hi[(w * kMaxProjPerPhase + j) * 16 + m];
        o.lo = S.red_lo[(w * kMaxProjPerPhase + j) * 16 + m];
        ss.add(o);
    }
}
__device__ __forceinline__ unsigned long long stats_word(float mx, const FF &ss, uint32_t tag) {
    const uint32_t mb = __float_as_uint(mx) >> 16;  // mx is a bf16 value: exact
    const uint32_t sb = __float_as_uint(ss.value());
    return static_cast<unsigned long long>(mb | (tag16_of(tag) << 16)) |
           (static_cast<unsigned long long>(sb) << 32);
}

__device__ __forceinline__ uint32_t quant1(float v, float c) {
    int iv = __float2int_rn(__fmul_rn(v, c));
    iv = iv > 127 ? 127 : (iv < -128 ? -128 : iv);
    return static_cast<uint32_t>(iv) & 0xffu;
}

// Metadata prefetch of one phase by one warp: issue (one round trip, 4
// words per lane) early, commit to shared memory late.
struct MetaLoad {
    uint32_t v[kMetaPerLane];
    __device__ __forceinline__ void issue(const Args &A, int p, int lane) {
        const uint32_t *src = reinterpret_cast<const uint32_t *>(A.metas + p);
#pragma unroll
        for (int u = 0; u < kMetaPerLane; ++u) {
            const int w = lane + 32 * u;
            v[u] = w < kMetaWords ? __ldg(src + w) : 0u;
        }
    }
    __device__ __forceinline__ void commit(const Shared &S, int p, int lane) const {
        uint32_t *dst = reinterpret_cast<uint32_t *>(&S.meta[p & 1]);
#pragma unroll
        for (int u = 0; u < kMetaPerLane; ++u) {
            const int w = lane + 32 * u;
            if (w < kMetaWords) dst[w] = v[u];
        }
    }
};

// ------------------------------------------------------------- producer --

// Ring of weight chunks (one per task), allocated first-in first-out in a
// byte ring so that small chunks do not waste space: the producer waits for
// the oldest chunks to be released until the new chunk fits.
__device__ void producer(const Args &A, const Shared &S) {
    const int cta = blockIdx.x;
    const uint32_t RB = A.ring_bytes;
    uint32_t idx = 0, tail = 0, head = 0;
    bool ok = true;
    for (int p = 0; p < A.nphase && ok; ++p) {
        // this phase's metadata in registers: all loads issued together
        const MetaImg &MI = A.metas[p];
        const Phase ph = MI.ph;
        const uint8_t *pk[kMaxProjPerPhase];
        int rb[kMaxProjPerPhase], re[kMaxProjPerPhase];
#pragma unroll
        for (int j = 0; j < kMaxProjPerPhase; ++j) {
            pk[j] = MI.pj[j].packed;
            rb[j] = MI.pj[j].rg_base;
            re[j] = MI.pj[j].rg_base + MI.pj[j].RG;
        }
        const Work w = work_of(ph, cta);
        if (!w.valid || w.npieces == 0) continue;
        const int ntask = w.nsets * w.npieces;
        const int64_t KT = ph.KT;
        for (int i = 0; i < ntask && ok; ++i) {
            const Task t = task_of(w, i);
            const uint32_t per = static_cast<uint32_t>(t.thi - t.tlo) * 512u;
            const uint32_t bytes = per * static_cast<uint32_t>(t.rhi - t.rlo);
            const uint32_t pos = head % RB;
            if (pos + bytes > RB) head += RB - pos;
            // free space: [head, coff[tail] + RB) once the chunks before tail are released
            while (ok && tail < idx && (idx - tail >= static_cast<uint32_t>(kDesc) ||
                                        head + bytes > S.coff[tail % kDesc] + RB)) {
                if (!mbar_wait_bounded(&S.empty[tail % kDesc], (tail / kDesc) & 1u, A.wait_limit) ||
                    *S.abort_flag)
                    ok = false;
                ++tail;
            }
            if (!ok) break;
            const uint32_t d = idx % kDesc;
            S.coff[d] = head;
            mbar_arrive_expect_tx(&S.full[d], bytes);
            uint8_t *dst = S.ring + head % RB;
            for (int r = t.rlo; r < t.rhi; ++r) {
                const uint8_t *base = pk[0];
                int rg0 = rb[0];
#pragma unroll
                for (int j = 1; j < kMaxProjPerPhase; ++j)
                    if (j < ph.nproj && r >= re[j - 1]) {
                        base = pk[j];
                        rg0 = rb[j];
                    }
                bulk_g2s(dst + (r - t.rlo) * per, base + (static_cast<int64_t>(r - rg0) * KT + t.tlo) * 512, per,
                         &S.full[d]);
            }
            head += bytes;
            ++idx;
        }
    }
    if (!ok) raise_abort(S, A.status);
    // Every copy issued must land before the CTA may exit.
    const uint32_t first = idx > static_cast<uint32_t>(kDesc) ? idx - kDesc : 0u;
    for (uint32_t k = first; k < idx; ++k)
        mbar_wait_bounded(&S.full[k % kDesc], (k / kDesc) & 1u, kDrainLimit);
}

// ------------------------------------------------------------- consumers -

template <int NT>
__device__ __forceinline__ void run_task(const Args &A, const Shared &S, const Phase &ph, const Work &w,
                                         const Task &t, uint32_t idx, int lane) {
    const int g = lane >> 2, tq = lane & 3;
    const int nrg = t.rhi - t.rlo;
    const uint32_t d = idx % kDesc;
    if (!mbar_wait_warp(&S.full[d], (idx / kDesc) & 1u, A.wait_limit)) {
        if (lane == 0) raise_abort(S, A.status);
        return;
    }
    const uint8_t *chunk = S.ring + S.coff[d] % A.ring_bytes;
    const uint32_t per = static_cast<uint32_t>(t.thi - t.tlo) * 512u;
    float acc[4][NT][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][j][e] = 0.0f;
    int corr[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) corr[j] = 0;
    const int qstride = ph.qstride;
    for (int kt = t.tlo; kt < t.thi; ++kt) {
        uint32_t b[NT][8][2];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const int tok = 8 * j + g;
            uint4 q0 = make_uint4(0, 0, 0, 0), q1 = q0;
            if (tok < A.M) {
                const uint8_t *src = S.qc + tok * qstride + (kt - w.t0) * 128 + tq * 32;
                q0 = *reinterpret_cast<const uint4 *>(src);
                q1 = *reinterpret_cast<const uint4 *>(src + 16);
            }
            dm::build_b(q0, q1, b[j], corr[j]);
        }
        const uint8_t *wt = chunk + (kt - t.tlo) * 512 + lane * 16;
        uint4 wv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) wv[i] = *reinterpret_cast<const uint4 *>(wt + (i < nrg ? i : 0) * per);
        dm::mma_tile<NT>(wv, b, acc);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[d]);
    // sum(q) per token: reduce over the four t lanes, then fetch this lane's tokens.
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        corr[j] += __shfl_xor_sync(0xffffffffu, corr[j], 1);
        corr[j] += __shfl_xor_sync(0xffffffffu, corr[j], 2);
    }
    const int Mp = A.Mp;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const int ce = __shfl_sync(0xffffffffu, corr[j], 4 * (2 * tq));
        const int co = __shfl_sync(0xffffffffu, corr[j], 4 * (2 * tq + 1));
        const int t0k = 8 * j + 2 * tq;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (i >= nrg) continue;
            int32_t *pr = S.part + ((t.rlo - w.r0 + i) * 16) * Mp;
            if (t0k < A.M) {
                atomicAdd(pr + g * Mp + t0k, __float2int_rn(acc[i][j][0] * 16777216.0f) - ce);
                atomicAdd(pr + (g + 8) * Mp + t0k, __float2int_rn(acc[i][j][2] * 16777216.0f) - ce);
            }
            if (t0k + 1 < A.M) {
                atomicAdd(pr + g * Mp + t0k + 1, __float2int_rn(acc[i][j][1] * 16777216.0f) - co);
                atomicAdd(pr + (g + 8) * Mp + t0k + 1, __float2int_rn(acc[i][j][3] * 16777216.0f) - co);
            }
        }
    }
}

template <int NT>
__device__ void consumers(const Args &A, const Shared &S) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x;
    const int M = A.M, Mp = A.Mp;
    const uint32_t epoch = *S.epoch;
    const uint32_t lim = A.wait_limit;

    for (int j = tid; j < A.nproj; j += kConsumers) S.gall[j] = __ldg(A.gammas[j]);
    if (warp == 1 && A.nphase > 0) {
        MetaLoad ml;
        ml.issue(A, 0, lane);
        ml.commit(S, 0, lane);
    }
    // ---- phase index 0: statistics of the chain input x over this CTA's k-range
    {
        const int chunks = A.K0 / 8;
        const int c0 = static_cast<int>(static_cast<int64_t>(cta) * chunks / A.nCTA);
        const int c1 = static_cast<int>(static_cast<int64_t>(cta + 1) * chunks / A.nCTA);
        float mx = 0.0f;
        FF ss;
        const int m = tid % Mp;
        for (int e = tid; e < (c1 - c0) * Mp; e += kConsumers) {
            if (m >= M) continue;
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(A.x + static_cast<int64_t>(m) * A.K0) + c0 + e / Mp);
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float a = __uint_as_float(wv[i] << 16), b = __uint_as_float(wv[i] & 0xffff0000u);
                mx = fmaxf(mx, fmaxf(fabsf(a), fabsf(b)));
                ss.add_sq(a);
                ss.add_sq(b);
            }
        }
        reduce_stats(S, 0, mx, ss, Mp, warp, lane);
        named_sync(1, kConsumers);
        if (tid < M) {
            float cm;
            FF cs;
            combine_stats(S, 0, tid, cm, cs);
            st_cg_u64(A.x_stats + cta * Mp + tid, stats_word(cm, cs, tag_of(epoch, 0)));
        }
        named_sync(1, kConsumers);
        if (tid == 0) red_relaxed_add_u32(A.ctl, 1u);
    }

    uint32_t chunk_base = 0;
    for (int p = 0; p < A.nphase; ++p) {
        const uint32_t tag = tag_of(epoch, p + 1);
        // ---- wait until every CTA finished the previous phase
        if (tid == 0) {
            const uint32_t target = static_cast<uint32_t>(p + 1) * static_cast<uint32_t>(A.nCTA);
            bool ok = false;
            for (uint32_t i = 0; i < lim; ++i) {
                if (ld_relaxed_u32(A.ctl) >= target) {
                    ok = true;
                    break;
                }
                if ((i & 63u) == 63u && (ld_relaxed_u32(A.status) & 1u) != 0u) break;
            }
            if (!ok) raise_abort(S, A.status);
        }
        if (named_sync_or(1, kConsumers, *S.abort_flag != 0)) break;
        const MetaImg &MT = S.meta[p & 1];
        const Phase ph = MT.ph;
        MetaLoad next;  // metadata of the next phase: fetched now, stored in the epilogue
        if (warp == 1 && p + 1 < A.nphase) next.issue(A, p + 1, lane);
        const Work w = work_of(ph, cta);

        // ---- statistics of the input: combine the producers' partials
        {
            const uint32_t want = tag16_of(tag_of(epoch, ph.in_phase));
            const int m = tid % Mp;
            const int n = A.nCTA * Mp;
            float mx = 0.0f;
            FF ss;
            bool ok = true;
            for (int e0 = tid; e0 < n; e0 += 12 * kConsumers) {
            unsigned long long v[12];
#pragma unroll
            for (int u = 0; u < 12; ++u) {
                const int e = e0 + u * kConsumers;
                if (e < n && m < M) v[u] = ld_cg_u64(ph.stats_in + e);
            }
#pragma unroll
            for (int u = 0; u < 12; ++u) {
                const int e = e0 + u * kConsumers;
                if (e >= n || m >= M) continue;
                if (!tag_ok(v[u], want, 0xffffu, 16)) {
                    v[u] = poll_tag(ph.stats_in + e, want, 0xffffu, 16, lim, A.status);
                    ok = ok && tag_ok(v[u], want, 0xffffu, 16);
                }
                mx = fmaxf(mx, __uint_as_float(static_cast<uint32_t>(v[u] & 0xffffu) << 16));
                ss.add(__uint_as_float(static_cast<uint32_t>(v[u] >> 32)));
            }
            }
            if (!ok) raise_abort(S, A.status);
            reduce_stats(S, 0, mx, ss, Mp, warp, lane);
            named_sync(1, kConsumers);
            if (tid < M) {
                float cm;
                FF cs;
                combine_stats(S, 0, tid, cm, cs);
                if (!(cm >= 1e-5f)) cm = 1e-5f;
                S.c[tid] = __fdiv_rn(127.0f, cm);
                // tok_scale = rms^-1 * max / 127, every step correctly rounded fp32
                const float ms = __fadd_rn(__fdiv_rn(cs.value(), static_cast<float>(ph.K)), A.eps);
                const float r = __fdiv_rn(1.0f, __fsqrt_rn(ms));
                S.ts[tid] = __fdiv_rn(__fmul_rn(r, cm), 127.0f);
            }
        }

        const bool has = w.valid && w.npieces > 0;
        if (has) {
            // ---- quantise this CTA's k-slice of the input into the q cache
            const int klo = w.t0 * 128, khi = min(w.t1 * 128, ph.K), kend = w.t1 * 128;
            const int qs = ph.qstride;
            named_sync(1, kConsumers);  // S.c ready
            bool ok = true;
            if (ph.act_in == nullptr) {
                const int per = (khi - klo) / 8;
                const int n = M * per;
                for (int e0 = tid; e0 < n; e0 += 8 * kConsumers) {
                    uint4 v[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int e = e0 + u * kConsumers;
                        if (e < n)
                            v[u] = __ldg(reinterpret_cast<const uint4 *>(A.x + static_cast<int64_t>(e / per) * ph.K +
                                                                         klo + 8 * (e % per)));
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int e = e0 + u * kConsumers;
                        if (e >= n) continue;
                        const int m = e / per, k = klo + 8 * (e % per);
                        const uint32_t wv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                        const float c = S.c[m];
                        uint32_t o[2] = {0u, 0u};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint32_t lo = quant1(__uint_as_float(wv[i] << 16), c);
                            const uint32_t hi = quant1(__uint_as_float(wv[i] & 0xffff0000u), c);
                            o[i >> 1] |= (lo | (hi << 8)) << (16 * (i & 1));
                        }
                        *reinterpret_cast<uint2 *>(S.qc + m * qs + (k - klo)) = make_uint2(o[0], o[1]);
                    }
                }
            } else {
                // pairs of tagged words (four values) per 16-byte load
                const uint32_t in_tag = tag_of(epoch, ph.in_phase);
                const int per = (khi - klo) / 4;
                const int half = ph.K / 2;
                const int n = M * per;
                for (int e0 = tid; e0 < n; e0 += 8 * kConsumers) {
                    ulonglong2 v[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int e = e0 + u * kConsumers;
                        if (e < n)
                            v[u] = ld_cg_u64x2(ph.act_in + static_cast<int64_t>(e / per) * half + klo / 2 + 2 * (e % per));
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int e = e0 + u * kConsumers;
                        if (e >= n) continue;
                        const int m = e / per, k = klo + 4 * (e % per);
                        const unsigned long long *src = ph.act_in + static_cast<int64_t>(m) * half + k / 2;
                        if (!tag_ok(v[u].x, in_tag, 0xffffffffu, 32)) {
                            v[u].x = poll_tag(src, in_tag, 0xffffffffu, 32, lim, A.status);
                            ok = ok && tag_ok(v[u].x, in_tag, 0xffffffffu, 32);
                        }
                        if (!tag_ok(v[u].y, in_tag, 0xffffffffu, 32)) {
                            v[u].y = poll_tag(src + 1, in_tag, 0xffffffffu, 32, lim, A.status);
                            ok = ok && tag_ok(v[u].y, in_tag, 0xffffffffu, 32);
                        }
                        const uint32_t b0 = static_cast<uint32_t>(v[u].x), b1 = static_cast<uint32_t>(v[u].y);
                        const float c = S.c[m];
                        const uint32_t q = quant1(__uint_as_float(b0 << 16), c) |
                                           (quant1(__uint_as_float(b0 & 0xffff0000u), c) << 8) |
                                           (quant1(__uint_as_float(b1 << 16), c) << 16) |
                                           (quant1(__uint_as_float(b1 & 0xffff0000u), c) << 24);
                        *reinterpret_cast<uint32_t *>(S.qc + m * qs + (k - klo)) = q;
                    }
                }
            }
            if (!ok) raise_abort(S, A.status);
            const int tail = kend - khi;  // k beyond K in the last tile reads as zero
            for (int e = tid; e < M * tail; e += kConsumers) S.qc[(e / tail) * qs + (khi - klo) + e % tail] = 0;
            for (int e = tid; e < w.nrgs * 16 * Mp; e += kConsumers) S.part[e] = 0;
        }
        if (named_sync_or(1, kConsumers, *S.abort_flag != 0)) break;

        // ---- tensor-core work on the streamed weight chunks
        if (has) {
            const int ntask = w.nsets * w.npieces;
            for (int i = warp; i < ntask; i += kConsumerWarps)
                run_task<NT>(A, S, ph, w, task_of(w, i), chunk_base + static_cast<uint32_t>(i), lane);
            chunk_base += static_cast<uint32_t>(ntask);
        }
        if (named_sync_or(1, kConsumers, *S.abort_flag != 0)) break;

        // ---- combine the K-split partial sums of the group
        int o0 = 0, o1 = 0;
        if (has) {
            o0 = w.s * w.nrgs / ph.S;
            o1 = (w.s + 1) * w.nrgs / ph.S;
            if (ph.S > 1) {
                const int n = w.nrgs * 16 * Mp;
                for (int e = tid; e < n; e += kConsumers) {
                    const int rl = e / (16 * Mp), m = e % Mp;
                    if ((rl >= o0 && rl < o1) || m >= M) continue;
                    const int row = (e / Mp) % 16;
                    const int64_t gi = ((static_cast<int64_t>(w.r0 + rl) * ph.S + w.s) * 16 + row) * Mp + m;
                    st_cg_u64(A.partials + gi, static_cast<unsigned long long>(static_cast<uint32_t>(S.part[e])) |
                                                        (static_cast<unsigned long long>(tag) << 32));
                }
                bool ok = true;
                const int own = (o1 - o0) * 16 * Mp;
                const int S1 = ph.S - 1;
                const int total = own * S1;  // (entry, peer) pairs
                // index of (owned entry, peer) pair f in the partial-sum buffer, or -1
                auto pidx = [&](int f) -> int64_t {
                    const int e = f / S1, k = f % S1, m = e % Mp;
                    if (f >= total || m >= M) return -1;
                    const int s2 = k < w.s ? k : k + 1;
                    const int rl = o0 + e / (16 * Mp), row = (e / Mp) % 16;
                    return ((static_cast<int64_t>(w.r0 + rl) * ph.S + s2) * 16 + row) * Mp + m;
                };
                for (int f0 = tid; f0 < total; f0 += 8 * kConsumers) {
                    unsigned long long v[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int64_t gi = pidx(f0 + u * kConsumers);
                        if (gi >= 0) v[u] = ld_cg_u64(A.partials + gi);
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int f = f0 + u * kConsumers;
                        const int64_t gi = pidx(f);
                        if (gi < 0) continue;
                        if (!tag_ok(v[u], tag, 0xffffffffu, 32)) {
                            v[u] = poll_tag(A.partials + gi, tag, 0xffffffffu, 32, lim, A.status);
                            ok = ok && tag_ok(v[u], tag, 0xffffffffu, 32);
                        }
                        atomicAdd(&S.part[o0 * 16 * Mp + f / S1], static_cast<int32_t>(static_cast<uint32_t>(v[u])));
                    }
                }
                if (!ok) raise_abort(S, A.status);
            }
        }
        if (named_sync_or(1, kConsumers, *S.abort_flag != 0)) break;

        // ---- epilogue: rescale, store, publish tagged outputs and statistics
        if (warp == 1 && p + 1 < A.nphase) next.commit(S, p + 1, lane);
        {
            const int m = tid % Mp;
            for (int j = 0; j < ph.nproj; ++j) {
                const Proj &P = MT.pj[j];
                float mx = 0.0f;
                FF ss;
                // owned local row groups of projection j
                const int lo = max(o0, P.rg_base - w.r0), hi = min(o1, P.rg_base + P.RG - w.r0);
                const int nent = hi > lo ? (hi - lo) * 8 * Mp : 0;
                const float f = __fmul_rn(S.gall[ph.proj0 + j], S.ts[m < M ? m : 0]);
                for (int e = tid; e < nent; e += kConsumers) {
                    if (m >= M) continue;
                    const int rp = (e / Mp) % 8, rl = lo + e / (8 * Mp);
                    const int n0 = (w.r0 + rl - P.rg_base) * 16 + 2 * rp;
                    uint32_t vb[2] = {0u, 0u};
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int n = n0 + h;
                        if (n >= P.N) continue;
                        const int32_t acc = S.part[(rl * 16 + 2 * rp + h) * Mp + m];
                        const __nv_bfloat16 v = __float2bfloat16_rn(__fmul_rn(static_cast<float>(acc), f));
                        const float vf = __bfloat162float(v);
                        vb[h] = static_cast<uint32_t>(__bfloat16_as_ushort(v));
                        if (P.out) P.out[static_cast<int64_t>(m) * P.N + n] = v;
                        if (P.acc_out) P.acc_out[static_cast<int64_t>(m) * P.N + n] = acc;
                        mx = fmaxf(mx, fabsf(vf));
                        ss.add_sq(vf);
                    }
                    if (P.act_out)
                        st_cg_u64(P.act_out + static_cast<int64_t>(m) * (P.N / 2) + n0 / 2,
                                       static_cast<unsigned long long>(vb[0] | (vb[1] << 16)) |
                                           (static_cast<unsigned long long>(tag) << 32));
                    if (w.r0 + rl == P.rg_base && rp == 0 && P.tok_scale_out) P.tok_scale_out[m] = S.ts[m];
                }
                reduce_stats(S, j, mx, ss, Mp, warp, lane);
            }
            named_sync(1, kConsumers);
            if (tid < ph.nproj * Mp) {
                const int j = tid / Mp, mm = tid % Mp;
                const Proj &P = MT.pj[j];
                if (mm < M && P.stats_out) {
                    float cm;
                    FF cs;
                    combine_stats(S, j, mm, cm, cs);
                    st_cg_u64(P.stats_out + cta * Mp + mm, stats_word(cm, cs, tag));
                }
            }
        }
        named_sync(1, kConsumers);
        if (tid == 0) red_relaxed_add_u32(A.ctl, 1u);
    }
}

template <int NT>
__global__ void __launch_bounds__(kThreads, 1) chain_kernel(const Args A) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const Shared S = carve(smem_raw, A);
    if (threadIdx.x == 0) {
        *S.abort_flag = 0;
        *S.epoch = ld_relaxed_u32(A.ctl + 2);
        for (int i = 0; i < kDesc; ++i) {
            mbar_init(&S.full[i], 1);
            mbar_init(&S.empty[i], 1);
        }
        mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x >= kConsumers) {
        if (threadIdx.x == kConsumers) producer(A, S);
    } else {
        consumers<NT>(A, S);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // The last CTA to leave resets the arrival counter and advances the
        // epoch for the next launch; no CTA reads the counter after its exit.
        const unsigned old = atomicAdd(A.ctl + 1, 1u);
        if (old == static_cast<unsigned>(A.nCTA) - 1u) {
            atomicExch(A.ctl, 0u);
            atomicExch(A.ctl + 1, 0u);
            atomicAdd(A.ctl + 2, 1u);
        }
    }
}

// -------------------------------------------------------------- host -----

struct HostPlan {
    std::vector<Phase> phases;
    std::vector<Proj> projs;
    int M = 0, Mp = 0, nCTA = 0, K0 = 0, NT = 1;
    uint32_t ring_bytes = 0, q_bytes = 0, part_bytes = 0;
    size_t off_phases = 0, off_projs = 0, off_xstats = 0, off_partials = 0, bytes = 0;
    std::vector<size_t> off_act, off_stats;  // per projection, 0 if not consumed
};

int g_force_split = 0;

inline size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// Choose the K-split of a phase: minimise an estimate of the phase's time
// on the slowest CTA (its weight bytes at its HBM share, its activation
// bytes at its L2 share, and the partial-sum exchange), within the
// shared-memory limits of the q cache and the partial sums.
int choose_split(int RGT, int KT, int Mp, int nCTA, uint32_t limit) {
    if (g_force_split > 0) {
        int S = g_force_split < KT ? g_force_split : KT;
        if (S > nCTA) S = nCTA;
        return S;
    }
    const int cands[] = {1, 2, 3, 4, 6, 8, 12, 16};
    int best = 0;
    double best_t = 1e30;
    for (int S : cands) {
        if (S > KT || S > nCTA) continue;
        const int G = nCTA / S;
        const int rg_max = (RGT + G - 1) / G;
        const int kt = (KT + S - 1) / S;
        const uint32_t qb = static_cast<uint32_t>(Mp) * (kt * 128 + 16);
        const uint32_t pb = static_cast<uint32_t>(rg_max) * 16 * Mp * 4;
        if (qb + pb > limit) continue;
        const double w_ns = rg_max * kt * 512.0 / 44.0;               // HBM share of one SM
        const double a_ns = Mp * kt * 128.0 * 4.0 / 100.0 + 150.0;     // tagged activations from L2
        const double x_ns = S > 1 ? 500.0 + rg_max * 16.0 * Mp * 8.0 * (S - 1) / S / 100.0 : 0.0;
        const double t = w_ns + a_ns + x_ns;
        if (t < best_t) {
            best_t = t;
            best = S;
        }
    }
    return best;
}

// Shared memory: the q cache and partial sums get what the per-block limit
// leaves beside the fixed arrays and a weight ring of at least kMinRing
// bytes; the ring then takes the rest, up to kMaxRing.
constexpr uint32_t kMinRing = 48 * 1024;
constexpr uint32_t kMaxRing = 160 * 1024;

int smem_optin() {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
    return v;
}

bitlinear_status_t build_plan(int64_t M, int64_t K0, const bitlinear_chain_proj_t *projs, int32_t nproj,
                              int nCTA, HostPlan &H) {
    if (M < 1 || M > 16 || K0 < 16 || (K0 % 16) != 0 || K0 > 65536) return BITLINEAR_ERR_INVALID_ARG;
    if (!projs || nproj < 1 || nproj > 4096) return BITLINEAR_ERR_INVALID_ARG;
    if (nCTA < 1 || nCTA > kMaxCTA) return BITLINEAR_ERR_UNSUPPORTED;
    if (nproj > kMaxProj) return BITLINEAR_ERR_UNSUPPORTED;
    const int smax = smem_optin();
    if (smax < static_cast<int>(smem_fixed_bytes() + kMinRing + 4096)) return BITLINEAR_ERR_UNSUPPORTED;
    const uint32_t qpart_limit = static_cast<uint32_t>(smax) - smem_fixed_bytes() - kMinRing - 1024;
    H = HostPlan();
    H.M = static_cast<int>(M);
    H.Mp = 1;
    while (H.Mp < H.M) H.Mp *= 2;
    H.nCTA = nCTA;
    H.K0 = static_cast<int>(K0);
    H.NT = M <= 8 ? 1 : 2;
    std::vector<int> width(nproj + 1);
    std::vector<bool> consumed(nproj + 1, false);
    width[0] = H.K0;
    for (int j = 0; j < nproj; ++j) {
        const bitlinear_chain_proj_t &P = projs[j];
        if (!P.packed || !P.gamma || P.N < 1 || P.N > (1 << 24) || P.input < 0 || P.input > j ||
            P.flags != 0)
            return BITLINEAR_ERR_INVALID_ARG;
        if (!aligned16(P.packed) || !aligned4(P.gamma) || (P.out_bf16 && !aligned16(P.out_bf16)) ||
            (P.acc_out && !aligned16(P.acc_out)) || (P.tok_scale_out && !aligned4(P.tok_scale_out)))
            return BITLINEAR_ERR_INVALID_ARG;
        width[j + 1] = static_cast<int>(P.N);
        consumed[P.input] = true;
    }
    for (int j = 0; j < nproj; ++j)
        if (consumed[j + 1] && ((width[j + 1] % 16) != 0 || width[j + 1] > 65536))
            return BITLINEAR_ERR_INVALID_ARG;  // becomes a K: multiple of 16, at most 65536
    // phases: consecutive projections reading the same input
    std::vector<int> phase_of(nproj);
    for (int j = 0; j < nproj; ++j) {
        const int in = projs[j].input;
        bool fresh = H.phases.empty();
        if (!fresh) {
            Phase &cur = H.phases.back();
            const int in_cur = projs[cur.proj0].input;
            fresh = in != in_cur || cur.nproj == kMaxProjPerPhase ||
                    (in > 0 && phase_of[in - 1] == static_cast<int>(H.phases.size()) - 1);
        }
        if (fresh) {
            Phase ph{};
            ph.proj0 = j;
            ph.nproj = 0;
            ph.K = width[in];
            ph.KT = (ph.K + 127) / 128;
            ph.in_phase = in == 0 ? 0 : phase_of[in - 1] + 1;
            H.phases.push_back(ph);
        }
        Phase &ph = H.phases.back();
        phase_of[j] = static_cast<int>(H.phases.size()) - 1;
        Proj pr{};
        pr.packed = projs[j].packed;
        pr.gamma = projs[j].gamma;
        pr.out = static_cast<__nv_bfloat16 *>(projs[j].out_bf16);
        pr.acc_out = projs[j].acc_out;
        pr.tok_scale_out = projs[j].tok_scale_out;
        pr.N = static_cast<int32_t>(projs[j].N);
        pr.RG = (pr.N + 15) / 16;
        pr.rg_base = ph.RGT;
        ph.RGT += pr.RG;
        ph.nproj += 1;
        H.projs.push_back(pr);
    }
    if (H.phases.size() > 1000) return BITLINEAR_ERR_UNSUPPORTED;
    // splits and limits
    uint64_t partial_words = 0;
    for (Phase &ph : H.phases) {
        const int S = choose_split(ph.RGT, ph.KT, H.Mp, nCTA, qpart_limit);
        if (S == 0) return BITLINEAR_ERR_UNSUPPORTED;
        ph.S = S;
        ph.G = nCTA / S;
        ph.rg_max = (ph.RGT + ph.G - 1) / ph.G;
        const int kt = (ph.KT + S - 1) / S;
        ph.qstride = kt * 128 + 16;
        H.q_bytes = std::max<uint32_t>(H.q_bytes, static_cast<uint32_t>(H.Mp * ph.qstride));
        H.part_bytes = std::max<uint32_t>(H.part_bytes, static_cast<uint32_t>(ph.rg_max * 16 * H.Mp * 4));
        if (S > 1)
            partial_words = std::max<uint64_t>(partial_words, static_cast<uint64_t>(ph.RGT) * S * 16 * H.Mp);
    }
    H.q_bytes = (H.q_bytes + 127) & ~127u;
    H.part_bytes = (H.part_bytes + 127) & ~127u;
    {
        const uint32_t room = static_cast<uint32_t>(smax) - smem_fixed_bytes() - H.q_bytes - H.part_bytes - 1024;
        H.ring_bytes = std::min(room, kMaxRing) & ~1023u;
    }
    // workspace layout: control words | phase metadata | gamma pointers | ...
    size_t off = 256;
    H.off_phases = off;
    off = align256(off + H.phases.size() * sizeof(MetaImg));
    H.off_projs = off;
    off = align256(off + H.projs.size() * sizeof(float *));
    H.off_xstats = off;
    off = align256(off + static_cast<size_t>(nCTA) * H.Mp * 8);
    H.off_act.assign(nproj, 0);
    H.off_stats.assign(nproj, 0);
    for (int j = 0; j < nproj; ++j) {
        if (!consumed[j + 1]) continue;
        H.off_stats[j] = off;
        off = align256(off + static_cast<size_t>(nCTA) * H.Mp * 8);
        H.off_act[j] = off;
        off = align256(off + static_cast<size_t>(H.M) * width[j + 1] * 4);
    }
    H.off_partials = off;
    off = align256(off + partial_words * 8);
    H.bytes = off;
    return BITLINEAR_OK;
}

// Device pointers of the plan, once the workspace base is known.
void bind_plan(HostPlan &H, uint8_t *ws, const bitlinear_chain_proj_t *projs, int32_t nproj) {
    for (int j = 0; j < nproj; ++j) {
        Proj &P = H.projs[j];
        P.act_out = H.off_act[j] ? reinterpret_cast<unsigned long long *>(ws + H.off_act[j]) : nullptr;
        P.stats_out = H.off_stats[j] ? reinterpret_cast<unsigned long long *>(ws + H.off_stats[j]) : nullptr;
    }
    for (Phase &ph : H.phases) {
        const int in = projs[ph.proj0].input;
        ph.act_in = in == 0 ? nullptr : reinterpret_cast<unsigned long long *>(ws + H.off_act[in - 1]);
        ph.stats_in = in == 0 ? reinterpret_cast<unsigned long long *>(ws + H.off_xstats)
                              : reinterpret_cast<unsigned long long *>(ws + H.off_stats[in - 1]);
    }
}

int sm_count() {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return v;
}

std::mutex g_attr_mutex;
bool g_attr_set[2][64] = {{false}};

template <int NT>
cudaError_t ensure_attr(uint32_t smem) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_attr_mutex);
    if (!g_attr_set[NT - 1][dev]) {
        int maxs = 0;
        e = cudaDeviceGetAttribute(&maxs, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(chain_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, maxs);
        if (e != cudaSuccess) return e;
        g_attr_set[NT - 1][dev] = true;
    }
    return cudaSuccess;
}

}  // namespace chain
}  // namespace bl

using namespace bl;

extern "C" size_t bitlinear_chain_workspace_bytes(int64_t M, int64_t K0, const bitlinear_chain_proj_t *projs,
                                                  int32_t nproj) {
    chain::HostPlan H;
    if (chain::build_plan(M, K0, projs, nproj, chain::sm_count(), H) != BITLINEAR_OK) return 0;
    return H.bytes;
}

extern "C" bitlinear_status_t bitlinear_chain_prepare(int64_t M, int64_t K0, const bitlinear_chain_proj_t *projs,
                                                      int32_t nproj, float eps, void *workspace,
                                                      size_t workspace_bytes, bitlinear_chain_plan_t *plan,
                                                      void *stream) {
    using namespace bl::chain;
    if (!plan || !workspace || !aligned16(workspace)) return BITLINEAR_ERR_INVALID_ARG;
    std::memset(plan, 0, sizeof(*plan));
    HostPlan H;
    const bitlinear_status_t st = build_plan(M, K0, projs, nproj, sm_count(), H);
    if (st != BITLINEAR_OK) return st;
    if (workspace_bytes < H.bytes) return BITLINEAR_ERR_INVALID_ARG;
    const uint32_t smem = smem_bytes_for(H.ring_bytes, H.q_bytes, H.part_bytes);
    int dev = 0, maxs = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&maxs, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return BITLINEAR_ERR_CUDA;
    if (smem > static_cast<uint32_t>(maxs)) return BITLINEAR_ERR_UNSUPPORTED;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    bind_plan(H, ws, projs, nproj);
    // one host image of the control words and the plan tables
    std::vector<uint8_t> img(H.off_xstats, 0);
    const uint32_t first_epoch = 1;  // tags of a cleared workspace (0) never match
    std::memcpy(img.data() + 8, &first_epoch, 4);
    for (size_t p = 0; p < H.phases.size(); ++p) {
        MetaImg mi{};
        mi.ph = H.phases[p];
        for (int j = 0; j < mi.ph.nproj; ++j) mi.pj[j] = H.projs[mi.ph.proj0 + j];
        std::memcpy(img.data() + H.off_phases + p * sizeof(MetaImg), &mi, sizeof(MetaImg));
    }
    for (size_t j = 0; j < H.projs.size(); ++j)
        std::memcpy(img.data() + H.off_projs + j * sizeof(float *), &H.projs[j].gamma, sizeof(float *));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, H.bytes, s) != cudaSuccess) return BITLINEAR_ERR_CUDA;
    if (cudaMemcpyAsync(ws, img.data(), img.size(), cudaMemcpyHostToDevice, s) != cudaSuccess)
        return BITLINEAR_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return BITLINEAR_ERR_CUDA;
    plan->workspace = workspace;
    plan->workspace_bytes = H.bytes;
    plan->M = M;
    plan->K0 = K0;
    plan->nphase = static_cast<int32_t>(H.phases.size());
    plan->nproj = nproj;
    plan->grid = H.nCTA;
    plan->threads = kThreads;
    plan->smem_bytes = static_cast<int32_t>(smem);
    plan->ring_bytes = H.ring_bytes;
    plan->q_bytes = H.q_bytes;
    plan->part_bytes = H.part_bytes;
    plan->mp = H.Mp;
    plan->eps = eps;
    plan->off_phases = H.off_phases;
    plan->off_projs = H.off_projs;
    plan->off_xstats = H.off_xstats;
    plan->off_partials = H.off_partials;
    plan->magic = kPlanMagic;
    return BITLINEAR_OK;
}

extern "C" bitlinear_status_t bitlinear_chain_run(const bitlinear_chain_plan_t *plan, const void *x_bf16,
                                                  void *stream) {
    using namespace bl::chain;
    if (!plan || plan->magic != kPlanMagic || !x_bf16 || !aligned16(x_bf16)) return BITLINEAR_ERR_INVALID_ARG;
    unsigned int *status = nullptr;
    if (bl::status_word(&status) != cudaSuccess) return BITLINEAR_ERR_CUDA;
    uint8_t *ws = static_cast<uint8_t *>(plan->workspace);
    Args A{};
    A.metas = reinterpret_cast<const MetaImg *>(ws + plan->off_phases);
    A.gammas = reinterpret_cast<const float *const *>(ws + plan->off_projs);
    A.nproj = plan->nproj;
    A.ring_bytes = plan->ring_bytes;
    A.x = static_cast<const __nv_bfloat16 *>(x_bf16);
    A.x_stats = reinterpret_cast<unsigned long long *>(ws + plan->off_xstats);
    A.partials = reinterpret_cast<unsigned long long *>(ws + plan->off_partials);
    A.ctl = reinterpret_cast<unsigned int *>(ws);
    A.status = status;
    A.nphase = plan->nphase;
    A.M = static_cast<int32_t>(plan->M);
    A.Mp = plan->mp;
    A.nCTA = plan->grid;
    A.K0 = static_cast<int32_t>(plan->K0);
    A.q_bytes = plan->q_bytes;
    A.part_bytes = plan->part_bytes;
    A.wait_limit = bl::current_wait_limit();
    A.eps = plan->eps;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(plan->grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(plan->smem_bytes);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (plan->M <= 8) {
        e = ensure_attr<1>(static_cast<uint32_t>(plan->smem_bytes));
        if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, chain_kernel<1>, A);
    } else {
        e = ensure_attr<2>(static_cast<uint32_t>(plan->smem_bytes));
        if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, chain_kernel<2>, A);
    }
    return e == cudaSuccess ? BITLINEAR_OK : BITLINEAR_ERR_CUDA;
}

extern "C" void bitlinear_chain_set_split(int32_t split) { bl::chain::g_force_split = split > 0 ? split : 0; }
