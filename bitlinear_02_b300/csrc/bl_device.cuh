// Device-side helpers shared by the BitLinear kernels (sm_103a only).
// Inline PTX wrappers for programmatic dependent launch, mbarriers,
// thread-block clusters and tcgen05 (TMEM allocation, MMA, loads).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../include/bitlinear.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ != 1030)
#error "bitlinear kernels are written for sm_103a only"
#endif

namespace bl {

// ---------------------------------------------------------------- host ---

uint32_t current_wait_limit();  // api.cu: spin limit of every bounded wait

// Validation helpers shared by the entry points.
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// ------------------------------------------------- debug bounds checks ---
//
// Built with -DBITLINEAR_DEBUG (libbitlinear_debug.so), every plain global
// load and store of the kernels is preceded by a check of its offset
// against its buffer's extent, stated apart from the index arithmetic that
// produced it: if (dbg_ok(offset fits, site)) access.  A failed check sets
// bit `site` of its translation unit's word and skips the access - no trap,
// so the context stays usable - and bitlinear_check_status collects every
// unit's word and reports BITLINEAR_ERR_BOUNDS.  Tensor-map (TMA) copies
// are bounds-checked by the hardware and need none.  In release builds
// dbg_ok is the constant true and the checks compile away.
#ifdef BITLINEAR_DEBUG
using DebugTake = cudaError_t (*)(unsigned int *, cudaStream_t);
void debug_register(DebugTake take, const char *unit);  // api.cu
static __device__ unsigned int g_dbg_bounds = 0u;       // one per translation unit
__device__ __forceinline__ bool dbg_ok(bool in_bounds, unsigned int site) {
    if (!in_bounds) atomicOr(&g_dbg_bounds, 1u << (site & 31u));
    return in_bounds;
}
// Reads and clears this unit's word (stream-ordered, then synchronised).
static cudaError_t dbg_take(unsigned int *v, cudaStream_t st) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(v, g_dbg_bounds, sizeof(unsigned int), 0, cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0u;
    e = cudaMemcpyToSymbolAsync(g_dbg_bounds, &zero, sizeof(unsigned int), 0, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(st);
}
namespace {
struct DebugUnit {
    DebugUnit() { debug_register(&dbg_take, __BASE_FILE__); }
} g_debug_unit;
}  // namespace
#else
__device__ __forceinline__ constexpr bool dbg_ok(bool, unsigned int) { return true; }
#endif
// Offset o (elements) of an access of n elements fits a buffer of `extent`.
__device__ __forceinline__ constexpr bool fits(int64_t o, int64_t n, int64_t extent) {
    return o >= 0 && o + n <= extent;
}

// Launch a kernel with programmatic dependent launch enabled (and an
// optional cluster shape).  The kernel itself decides when it may start
// reading data produced by the previous kernel in the stream
// (griddepcontrol.wait) and when its dependents may launch.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, unsigned cluster_x, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    int n = 0;
    attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster_x > 1) {
        attrs[n].id = cudaLaunchAttributeClusterDimension;
        attrs[n].val.clusterDim.x = cluster_x;
        attrs[n].val.clusterDim.y = 1;
        attrs[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ------------------------------------------------------------- device ---

// Programmatic dependent launch: let the next kernel in the stream launch
// now / wait until the previous kernel's results are visible.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Streaming 16-byte load that does not allocate in L1 (weights: read once).
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
// Cached read-only 16-byte load (activations: reused by many CTAs).
__device__ __forceinline__ uint4 ld_ro16(const void *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t hadd2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// ---- mbarrier (CTA scope) ----
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("{.reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0];}" ::"r"(smem_addr(bar))
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{.reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p;}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: returns false (and the caller records a timeout) after
// `limit` unsuccessful tries instead of spinning forever.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// Bounded wait of one thread that also gives up as soon as another role of
// the CTA has raised the shared abort flag; a wait that expires raises it.
// So one expired wait ends every role's waits within a few polls, instead
// of each role spinning through its own limit.
__device__ __forceinline__ bool mbar_wait_abortable(uint64_t *bar, uint32_t parity, uint32_t limit,
                                                    volatile int *abort) {
    for (uint32_t i = 0; i < limit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
    }
    *abort = 1;
    return false;
}
// The same for a whole warp (every lane calls it; the outcome is the same in
// every lane, so the warp stays converged for .sync.aligned instructions).
__device__ __forceinline__ bool mbar_wait_abortable_warp(uint64_t *bar, uint32_t parity, uint32_t limit,
                                                         volatile int *abort) {
    for (uint32_t i = 0; i < limit; ++i) {
        if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
        if (__any_sync(0xffffffffu, *abort != 0)) return false;
    }
    *abort = 1;
    return false;
}

// Arrive on an mbarrier and add `bytes` to the transaction count it waits for.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

// ---- L2-only accesses (statistics exchanged between CTAs) ----
// Bulk prefetch of a global range into L2 (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ unsigned ld_cg_u32(const void *p) {
    unsigned v;
    asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ float ld_cg_f32(const void *p) { return __uint_as_float(ld_cg_u32(p)); }


__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- clusters ----
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}
__device__ __forceinline__ uint32_t cluster_map(uint32_t local_smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_smem_addr), "r"(rank));
    return r;
}
__device__ __forceinline__ int ld_cluster_s32(uint32_t addr) {
    int v;
    asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
// Four consecutive 32-bit words of a cluster peer's shared memory (16-byte aligned).
__device__ __forceinline__ int4 ld_cluster_v4(uint32_t addr) {
    int4 v;
    asm volatile("ld.shared::cluster.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}
__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// ---- tcgen05 (1-CTA group) ----
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16, fp32 accumulate; A is
// 128 rows (lanes) x 16 f16 (8 columns, two f16 per column) in tensor memory.
__device__ __forceinline__ void tc_mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{.reg .pred p; setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns from 16 registers per thread.
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
// One lane of a converged warp (elect.sync): the lane that issues the
// warp's single-thread tcgen05 operations.
__device__ __forceinline__ bool elect_one() {
    uint32_t p;
    asm volatile("{.reg .pred P; .reg .b32 r; elect.sync r|P, 0xffffffff; selp.u32 %0, 1, 0, P;}" : "=r"(p));
    return p != 0;
}
__device__ __forceinline__ void tc_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// Arrive on an mbarrier once all previously issued tcgen05.mma of this
// thread have completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(bar))
        : "memory");
}
__device__ __forceinline__ void tc_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile stored with
// the 128-byte swizzle: rows of 64 f16 (128 B), 8-row atoms of 1024 B.
// Fields: start address >> 4 (bits 0-13), leading byte offset >> 4
// (16-29, unused for this layout), stride byte offset >> 4 (32-45: 1024 B
// between 8-row atoms), descriptor version 1 (46-47), swizzle mode
// 128B = 2 (61-63).  The tile must start on a 1024-byte boundary.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(1u) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}
// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` in such a tile.
__device__ __forceinline__ uint32_t sw128_off(uint32_t row, uint32_t chunk) {
    return (row >> 3) * 1024u + (row & 7u) * 128u + ((chunk ^ (row & 7u)) << 4);
}
// Instruction descriptor, kind::f16: D fp32, A and B f16, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32(uint32_t M, uint32_t N) {
    return (1u << 4)                 // D format: f32
           | (0u << 7) | (0u << 10)  // A, B format: f16
           | ((N >> 3) << 17) | ((M >> 4) << 24);
}

}  // namespace bl
