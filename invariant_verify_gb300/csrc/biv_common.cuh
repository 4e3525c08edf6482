// Internal helpers shared by the libbiv translation units: host-side status
// plumbing, and device-side inline PTX for mbarriers, TMA, tcgen05 and
// bounded waits.  Written for sm_103a (GB300) only.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <nvtx3/nvToolsExt.h>

#include "../../include/biv.h"

#define BIV_DEV __device__ __forceinline__

// Host-side trace range named after the ABI call (NVTX; a pointer check when no
// tool is attached, so ncu can take `--nvtx --nvtx-include <call>/` to capture
// one call's kernels).  Under stream capture it marks the enqueue.
struct BivTraceScope {
    explicit BivTraceScope(const char* name) { nvtxRangePushA(name); }
    ~BivTraceScope() { nvtxRangePop(); }
    BivTraceScope(const BivTraceScope&) = delete;
    BivTraceScope& operator=(const BivTraceScope&) = delete;
};
#define BIV_TRACE_CALL() const BivTraceScope biv_trace_scope_(__func__)

namespace biv {

// ------------------------------------------------------------------ host
void set_cuda_error(cudaError_t e);                 // thread-local record (biv_api.cpp)
inline int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return BIV_OK;
    set_cuda_error(e);
    return BIV_ERR_CUDA;
}
inline int launch_status() { return cuda_status(cudaGetLastError()); }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int num_sms();                                      // of the current device, cached

// Per-device one-time set-up (kernel attributes, symbol addresses), safe to
// call from several host threads: run(dev, f) calls f() until it returns
// BIV_OK once for that device, and returns BIV_OK without calling it after.
constexpr int kMaxDevices = 64;
struct DeviceOnce {
    std::mutex mu;
    bool done[kMaxDevices] = {};
    template <typename F>
    int run(int dev, F&& f) {
        if (dev < 0 || dev >= kMaxDevices) return BIV_ERR_DEVICE;
        std::lock_guard<std::mutex> lock(mu);
        if (done[dev]) return BIV_OK;
        const int st = f();
        if (st == BIV_OK) done[dev] = true;
        return st;
    }
};

// cuTensorMapEncodeTiled from the driver (through the runtime's entry-point
// query, so no link against libcuda); null if unavailable.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn();

// Launch with programmatic dependent launch: the kernel may start while the
// previous kernel on the stream is finishing; it must execute pdl_wait()
// before its first global-memory access.  Captured launches keep the
// programmatic edge inside CUDA graphs.
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
               Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...));
}

// The same for a kernel launched in clusters of `cluster_x` CTAs along x.
template <typename... KArgs, typename... Args>
int launch_cluster_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       int cluster_x, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(cluster_x);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cuda_status(cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...));
}

// Each translation unit owns one device error word and registers a reader.
typedef cudaError_t (*err_reader_fn)(uint32_t* bits, bool clear);
void register_err_reader(err_reader_fn fn);

#define BIV_DEFINE_ERR_WORD(NAME)                                                            \
    static __device__ unsigned int NAME;                                                     \
    static cudaError_t NAME##_read(uint32_t* bits, bool clear) {                            \
        unsigned int v = 0;                                                                  \
        cudaError_t e = cudaMemcpyFromSymbol(&v, NAME, sizeof(v));                           \
        if (e != cudaSuccess) return e;                                                      \
        *bits |= v;                                                                          \
        if (clear && v) {                                                                    \
            unsigned int z = 0;                                                              \
            e = cudaMemcpyToSymbol(NAME, &z, sizeof(z));                                     \
        }                                                                                    \
        return e;                                                                            \
    }                                                                                        \
    static struct NAME##_reg_t {                                                             \
        NAME##_reg_t() { ::biv::register_err_reader(&NAME##_read); }                         \
    } NAME##_reg;

// ---------------------------------------------------------------- device
constexpr unsigned long long kWaitLimitNs = 2000000000ull;   // 2 s bound on any spin

BIV_DEV uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Programmatic dependent launch: wait until the preceding kernel of the
// stream has completed and its writes are visible (a no-op when the kernel
// was launched without a programmatic dependency), and let the next kernel
// begin launching.
BIV_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
BIV_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

BIV_DEV uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

BIV_DEV void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (TMA, tensor-core operand reads).
BIV_DEV void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

BIV_DEV void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

BIV_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

BIV_DEV void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

BIV_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking probe of a phase: never suspends the thread.
BIV_DEV bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

BIV_DEV bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity);

// Wait for the phase of `bar` with the given parity to complete, for at most
// about kWaitLimitNs.  The first kFastPolls polls touch nothing but the
// barrier (reading the global timer is slow); only a wait that outlasts them
// starts the clock.  On time-out: raise BIV_DEVERR_TIMEOUT in *err, set the
// CTA's abort flag (shared memory) and return false.  Also returns false as
// soon as another thread of the CTA has aborted.
constexpr int kFastPolls = 4096;

// spin = true polls with test_wait (no suspension: the single producer / MMA
// threads of a pipeline react at once); spin = false uses try_wait, which may
// park the thread until the phase completes (for warps that wait long).
// cluster = true: try_wait with acquire at cluster scope, for a barrier that
// threads of another CTA of the cluster arrive on.
BIV_DEV bool mbar_poll(uint64_t* bar, uint32_t parity, bool spin, bool cluster) {
    return cluster ? mbar_try_wait_cluster(bar, parity)
                   : (spin ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity));
}

BIV_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, unsigned int* err,
                       bool spin = false, bool cluster = false) {
#pragma unroll 1
    for (int i = 0; i < kFastPolls; ++i)
        if (mbar_poll(bar, parity, spin, cluster)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
        for (int i = 0; i < 256; ++i)
            if (mbar_poll(bar, parity, spin, cluster)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            atomicOr(err, BIV_DEVERR_TIMEOUT);
            return false;
        }
    }
}

// Wait without abort propagation (used only while draining after an abort).
BIV_DEV bool mbar_wait_drain(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > kWaitLimitNs) return false;
    }
    return true;
}

// 2-D tiled TMA load global -> shared, completion counted on `bar` in bytes.
// c0 is the innermost (contiguous) coordinate in elements.
BIV_DEV void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                         uint64_t cache_policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(cache_policy)
        : "memory");
}

// 3-D tiled TMA load (coordinates innermost first), completion on `bar`.
BIV_DEV void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2,
                         uint64_t cache_policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(cache_policy)
        : "memory");
}

// Prefetch one 3-D tiled box into L2 (no shared memory, no completion).
BIV_DEV void tma_prefetch_3d(const CUtensorMap* map, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

// 4-D tiled TMA load (coordinates innermost first), completion on `bar`.
BIV_DEV void tma_load_4d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2, int c3,
                         uint64_t cache_policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar)),
        "l"(cache_policy)
        : "memory");
}

BIV_DEV void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

BIV_DEV uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

BIV_DEV uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ------------------------------------------------------------ clusters
// Rank of this CTA in its cluster.
BIV_DEV uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Execution and memory barrier over every thread of every CTA of the cluster
// (the non-aligned form: the threads of a warp may arrive apart).
BIV_DEV void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// The shared::cluster address of `p` (a shared variable of this CTA) in the
// shared memory of the cluster's CTA `rank` (the same variable there).
BIV_DEV uint32_t mapa_shared(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

// Arrive once on an mbarrier of any CTA of the cluster (shared::cluster
// address), releasing this thread's prior writes at cluster scope.
BIV_DEV void mbar_arrive_cluster(uint32_t bar_cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster_addr) : "memory");
}

// Phase probe with acquire at cluster scope (for barriers other CTAs of the
// cluster arrive on).
BIV_DEV bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// 3-D tiled TMA load into this CTA's shared memory whose completion is
// counted on an mbarrier of either CTA of the pair (shared::cluster address):
// the loads of both CTAs of a pair feed the even CTA's barrier.
BIV_DEV void tma_load_3d_pair(void* smem_dst, const CUtensorMap* map, uint32_t bar_cluster_addr, int c0, int c1,
                              int c2, uint64_t cache_policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar_cluster_addr), "l"(cache_policy)
        : "memory");
}

// ------------------------------------------------------------- tcgen05
BIV_DEV void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

BIV_DEV void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

BIV_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// The same for a CTA pair (cta_group::2): one warp of each CTA of the pair
// executes these together; the columns are allocated at the same address in
// both CTAs' tensor memory.
BIV_DEV void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

BIV_DEV void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

BIV_DEV void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

BIV_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
BIV_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D(tmem) (+)= A(smem) * B(smem)^T, bf16 inputs, fp32 accumulate, one CTA.
BIV_DEV void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The same MMA issued by one elected lane of a converged warp whose lanes all
// hold the same operands (the warp-uniform form issues faster than a lone
// thread).
BIV_DEV void umma_bf16_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D (+)= A * B^T across a CTA pair (cta_group::2, M = 256): rows 0..127 of A
// come from the even CTA's shared memory and rows 128..255 from the odd
// CTA's, at the same address; likewise the first and second halves of B's N
// rows.  Each CTA's tensor memory receives its own 128 rows of D.  Issued by
// one elected lane of the even CTA.
BIV_DEV void umma_bf16_pair_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                  uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on an mbarrier of either CTA of the pair (shared::cluster
// address) when the pair MMAs issued so far by this thread complete.
BIV_DEV void umma_commit_pair_elect(uint32_t bar_cluster_addr) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}\n" ::"r"(
            bar_cluster_addr)
        : "memory");
}

// tcgen05.commit by the elected lane (the lane that issued the MMAs above).
BIV_DEV void umma_commit_elect(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}\n" ::"r"(
            smem_u32(bar))
        : "memory");
}

// Arrive once on `bar` when all previously issued tcgen05.mma of this thread complete.
BIV_DEV void umma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

BIV_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 lanes x 16 consecutive 32-bit columns: thread t gets lane (base lane + t).
BIV_DEV void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// 32 lanes x 32 consecutive 32-bit columns, and the wait for it in the same
// statement (the registers are only read after the load has completed).
BIV_DEV void tmem_ld32_sync(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
          "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// M = 64 accumulators (lanes 0..15 of each 32-lane quarter): threads 0..15 get
// their lane's columns [c, c + 16), threads 16..31 the same lanes' columns
// [c + 16, c + 32); the wait is in the same statement.
BIV_DEV void tmem_ld16x2_sync(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16], 16;\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// The same load without its wait: several may be in flight before one
// tmem_ld_wait(), after which reg_fence16 on each destination keeps every use
// of the registers behind the wait.
BIV_DEV void tmem_ld16x2(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16], 16;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
// Eight 32-bit words to global memory in one 32-byte store (p 32-byte aligned):
// a whole sector per thread where a row-per-lane layout scatters a warp's
// stores over many rows.
BIV_DEV void st_global_v8(void* p, const uint32_t* v) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]), "r"(v[1]),
                 "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

BIV_DEV void reg_fence16(uint32_t (&r)[16]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                   "+r"(r[14]), "+r"(r[15]));
}

// Shared-memory matrix descriptor for a K-major bf16 tile written by TMA with
// 128-byte swizzle: rows of 128 B (64 bf16 along K), 8-row atoms 1024 B apart.
// Start address in 16-B units (bits 0-13), leading offset unused for swizzled
// K-major (1), stride offset 1024 B (bits 32-45), descriptor version 1
// (bits 46-47), swizzle mode 2 = 128 B (bits 61-63).
BIV_DEV uint64_t sw128_kmajor_desc(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1u) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), bf16 A
// and B (bits 7-9, 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 in bits
// 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// 2^x by the hardware approximation (ex2.approx, subnormal results flushed).
BIV_DEV float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ------------------------------------------------------------ bf16 pack
BIV_DEV uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

BIV_DEV float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
BIV_DEV float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// SiLU(g) = g / (1 + e^-g), one definition for every kernel that applies it
// (the SwiGLU kernel and the gate/up GEMM epilogue give the same bits).
BIV_DEV float silu(float g) { return __fdiv_rn(g, __fadd_rn(1.0f, expf(-g))); }

// bf16(silu(g) * u) of two bf16 values packed as (lo, hi) pairs.
BIV_DEV uint32_t swiglu_pack(uint32_t g2, uint32_t u2) {
    return pack_bf16x2(__fmul_rn(silu(bf16lo(g2)), bf16lo(u2)), __fmul_rn(silu(bf16hi(g2)), bf16hi(u2)));
}

// Rotate-half RoPE of the pair (a, b) = (x[i], x[i + hd/2]) of one head by the
// angle pos * theta^(-2i/hd); one definition for every kernel that rotates
// (the RoPE kernels and the QKV GEMM's RoPE epilogue), so all give the same
// bits.  Explicit roundings: no fma contraction.
// Rotation frequency theta^(-2i/hd) of RoPE pair i.
BIV_DEV float rope_inv_freq(int i, int hd, float theta) {
    return powf(theta, -2.0f * static_cast<float>(i) / static_cast<float>(hd));
}

// The rotation angle of pair frequency inv_freq at position pos, as sine and cosine.
BIV_DEV void rope_sincos(int pos, float inv_freq, float& sn, float& cs) {
    const float ang = __fmul_rn(static_cast<float>(pos), inv_freq);
    sincosf(ang, &sn, &cs);
}

// One RoPE pair (a, b) rotated by the angle with the given sine and cosine.
BIV_DEV void rope_rotate(float a, float b, float sn, float cs, __nv_bfloat16& o1, __nv_bfloat16& o2) {
    o1 = __float2bfloat16_rn(__fsub_rn(__fmul_rn(a, cs), __fmul_rn(b, sn)));
    o2 = __float2bfloat16_rn(__fadd_rn(__fmul_rn(b, cs), __fmul_rn(a, sn)));
}

// One RoPE pair (a, b) at position pos with the pair's frequency given.
BIV_DEV void rope_pair_f(float a, float b, int pos, float inv_freq, __nv_bfloat16& o1, __nv_bfloat16& o2) {
    float sn, cs;
    rope_sincos(pos, inv_freq, sn, cs);
    rope_rotate(a, b, sn, cs, o1, o2);
}

BIV_DEV void rope_pair(float a, float b, int pos, int i, int hd, float theta, __nv_bfloat16& o1,
                       __nv_bfloat16& o2) {
    rope_pair_f(a, b, pos, rope_inv_freq(i, hd, theta), o1, o2);
}

// M = 64 accumulators, two loads and one wait: threads 0..15 get their lane's
// columns [a, a + N) and [b, b + N), threads 16..31 the same lanes' columns
// [a + N, a + 2N) and [b + N, b + 2N) (N = 4 or 8).
BIV_DEV void tmem_ld16x2_x4_pair_sync(uint32_t ta, uint32_t tb, uint32_t (&a)[4], uint32_t (&b)[4]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x32bx2.x4.b32 {%0, %1, %2, %3}, [%8], 4;\n\t"
        "tcgen05.ld.sync.aligned.16x32bx2.x4.b32 {%4, %5, %6, %7}, [%9], 4;\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3])
        : "r"(ta), "r"(tb)
        : "memory");
}
BIV_DEV void tmem_ld16x2_x8_pair_sync(uint32_t ta, uint32_t tb, uint32_t (&a)[8], uint32_t (&b)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x32bx2.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%16], 8;\n\t"
        "tcgen05.ld.sync.aligned.16x32bx2.x8.b32 {%8, %9, %10, %11, %12, %13, %14, %15}, [%17], 8;\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]),
          "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7])
        : "r"(ta), "r"(tb)
        : "memory");
}

BIV_DEV void rope_rotate(float a, float b, int pos, int i, int hd, float theta, __nv_bfloat16* o1,
                         __nv_bfloat16* o2) {
    rope_pair(a, b, pos, i, hd, theta, *o1, *o2);
}

}  // namespace biv
