// common.cuh -- shared device primitives for the sm_103a kernels: inline
// PTX for mbarriers, TMA (cp.async.bulk.tensor), tcgen05 (TMEM alloc, UMMA,
// commit, TMEM loads), bounded waits, and the monotonic float key used by
// the max reductions.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "../../include/mc_max.h"

#define MC_HD __host__ __device__ __forceinline__
#define MC_D __device__ __forceinline__

namespace mc {

// ---------------------------------------------------------------------------
// monotonic float <-> uint32 key: key(a) < key(b)  <=>  a < b for all
// non-NaN floats, every NaN maps to the largest key, and key 0 lies below
// every float (it marks "no value yet").
// ---------------------------------------------------------------------------
MC_HD uint32_t float_key(float f) {
    uint32_t u;
#ifdef __CUDA_ARCH__
    u = __float_as_uint(f);
#else
    memcpy(&u, &f, 4);
#endif
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0xFFFFFFFFu;  // NaN
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
MC_HD float key_float(uint32_t k) {
    uint32_t u;
    if (k == 0xFFFFFFFFu) u = 0x7FC00000u;  // canonical NaN
    else u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    float f;
#ifdef __CUDA_ARCH__
    f = __uint_as_float(u);
#else
    memcpy(&f, &u, 4);
#endif
    return f;
}

#ifdef __CUDACC__

// ---------------------------------------------------------------------------
// programmatic dependent launch: every library kernel is launched with
// programmatic stream serialization, so its launch and prologue overlap the
// tail of the previous kernel on the stream.  pdl_wait() blocks until that
// kernel has completed and its writes are visible (it precedes every global
// access); pdl_trigger() lets the next kernel start its prologue.
// ---------------------------------------------------------------------------
MC_D void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MC_D void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
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
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// ---------------------------------------------------------------------------
// status word
// ---------------------------------------------------------------------------
MC_D void set_status(unsigned* status, unsigned bits) {
    if (status) atomicOr(status, bits);
}

MC_D uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// every on-chip wait gives up after this long and flags MC_DEV_TIMEOUT
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s

// ---------------------------------------------------------------------------
// shared memory / mbarrier
// ---------------------------------------------------------------------------
MC_D uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

MC_D void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
MC_D void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
MC_D void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
MC_D void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
MC_D bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on an mbarrier phase.  Returns false (and flags the status
// word and the CTA's abort flag) when the limit expires or another role of
// the CTA has already aborted.
MC_D bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, unsigned* status,
                    uint64_t limit_ns = kWaitLimitNs) {
    uint32_t b = smem_u32(bar);
    if (mbar_try_wait(b, parity)) return true;
    uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(b, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            set_status(status, MC_DEV_TIMEOUT);
            return false;
        }
    }
}

// ---------------------------------------------------------------------------
// TMA
// ---------------------------------------------------------------------------
MC_D void tma_load_3d(void* dst, const CUtensorMap* tm, uint64_t* bar, int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
// Pair load: the copy lands in this CTA's shared memory and completes on the
// mbarrier at cluster address bar (the even CTA's, for both CTAs of a pair).
MC_D void tma_load_3d_pair(void* dst, const CUtensorMap* tm, uint32_t bar, int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
// Tiled TMA store shared -> global of one box at (c0, c1, c2), tracked by the
// issuing thread's bulk async-group; elements outside the tensor are skipped.
MC_D void tma_store_3d(const CUtensorMap* tm, const void* src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(tm)),
                 "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}
MC_D void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the shared-memory sources of this thread's bulk copies have been read
MC_D void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// this thread's bulk copies have completed their global writes
MC_D void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// generic-proxy shared-memory writes -> visible to the async proxy (bulk copies)
MC_D void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
MC_D void tma_prefetch_desc(const CUtensorMap* tm) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05
// ---------------------------------------------------------------------------
MC_D void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
MC_D void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
MC_D void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
// CTA pairs (cluster of 2, cta_group::2): TMEM allocated collectively by one
// warp of each CTA at the same address; MMAs issued by the even CTA work on
// both CTAs' shared memory and TMEM.
MC_D void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
MC_D void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
MC_D void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
MC_D uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// shared::cluster address of the variable at shared address a in CTA `rank`
MC_D uint32_t mapa_shared(uint32_t a, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
MC_D void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// all threads of both CTAs of the cluster (start-up and teardown only)
MC_D void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
MC_D void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MC_D void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulate)
MC_D void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                    uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive on `bar` once every tcgen05 op issued so far by this thread is done
MC_D void umma_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive on the barrier at this shared offset in both CTAs of the pair once
// the pair MMAs issued so far by this thread have completed
MC_D void umma_commit_pair_both(uint64_t* bar) {
    const uint16_t mask = 3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(mask)
        : "memory");
}
MC_D void umma_commit_pair(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
MC_D void umma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i gets lane (base + i)
MC_D void tmem_ld32(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
        "[%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}
MC_D void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 format:
// start>>4 in [0,14), LBO>>4 in [16,30), SBO>>4 in [32,46), version 1 at
// bit 46, swizzle mode 2 (128B) in [61,64)).
MC_D uint64_t sw128_desc(uint32_t smem_addr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16: D f32; A and B both bf16 (f16 = 0) or
// both fp16 (f16 = 1); A K-major; B K-major (b_mn = 0) or MN-major
// (b_mn = 1); shape M x N.
MC_HD uint32_t idesc_f16kind(int M, int N, int b_mn, int f16) {
    const uint32_t ab = f16 ? 0u : 1u;
    return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// three-input max that returns NaN when any input is NaN
MC_D float max3_nan(float a, float b, float c) {
    float d;
    asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
MC_D float max_nan(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

MC_D float warp_max_nan(float v) {
    for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// Max-merge of v into *addr in the float order with NaN above +inf: values
// with the sign bit clear compare as signed integers, values with it set as
// reversed unsigned integers, so one integer atomic merges each value.
// *addr holds a float or the pattern 0xFFFFFFFF, which sorts below every
// value; NaN is merged as the canonical positive NaN.
MC_D void atomic_max_float(float* addr, float v) {
    uint32_t u = __float_as_uint(v);
    if (isnan(v)) u = 0x7FFFFFFFu;
    if (u & 0x80000000u) atomicMin(reinterpret_cast<unsigned*>(addr), u);
    else atomicMax(reinterpret_cast<int*>(addr), (int)u);
}

// A work item's raw maximum m merged into S_max[h], and into S_max[b, h]
// when s_bh is given, as S = m / sqrt(d): the division is monotonic, so the
// merged value is the maximum logit over the items divided once.  A
// non-finite S sets the status bit.
MC_D void merge_smax(float m, float sqrt_d, float* s_max, float* s_bh, int b, int H, int h, unsigned* status) {
    const float s = __fdiv_rn(m, sqrt_d);
    if (!isfinite(s)) set_status(status, MC_DEV_NONFINITE);
    atomic_max_float(s_max + h, s);
    if (s_bh) atomic_max_float(s_bh + (size_t)b * H + h, s);
}

// S_max[h] = max over sequences of key / sqrt(d) (NaN propagates); the
// per-sequence maxima are written too when s_bh is given.
MC_D void finalize_head(const unsigned* keys, int B, int H, int h, float sqrt_d, int accumulate,
                        float* s_max, float* s_bh, unsigned* status) {
    unsigned best = 0;
    for (int b = 0; b < B; ++b) {
        unsigned k = __ldcg(keys + b * H + h);
        if (s_bh) s_bh[b * H + h] = __fdiv_rn(key_float(k), sqrt_d);
        best = max(best, k);
    }
    float s = __fdiv_rn(key_float(best), sqrt_d);
    if (accumulate) s = max_nan(s_max[h], s);
    if (!isfinite(s)) set_status(status, MC_DEV_NONFINITE);
    s_max[h] = s;
}

// 32 lanes x 32 consecutive 32-bit columns from registers: thread i writes
// lane (base + i); tmem_st_wait() before the columns are read or reused
MC_D void tmem_st32(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns
MC_D void tmem_st16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
MC_D void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

#endif  // __CUDACC__

}  // namespace mc
