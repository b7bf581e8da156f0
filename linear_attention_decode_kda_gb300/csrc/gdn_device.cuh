// Device helpers shared by the step kernels: input loads, the scalar maps of
// the step, programmatic dependent launch, thread-block clusters, mbarriers
// and TMA bulk copies (inline PTX for sm_100+ / sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {
namespace dev {

__device__ __forceinline__ float ld_in(const void *p, size_t i, int bf16)
{
    if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[i]);
    return reinterpret_cast<const float *>(p)[i];
}

__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }
__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + expf(-x)); }
__device__ __forceinline__ float softplus_f(float x)
{
    return fmaxf(x, 0.0f) + log1pf(expf(-fabsf(x)));
}

// 4-tap causal conv: taps 0..2 on the kept window (oldest first), tap 3 on x.
__device__ __forceinline__ float conv4_silu(const float4 w, const float *win, float x)
{
    float acc = w.x * win[0];
    acc = fmaf(w.y, win[1], acc);
    acc = fmaf(w.z, win[2], acc);
    acc = fmaf(w.w, x, acc);
    return silu_f(acc);
}

// The same maps on the hardware exponential, logarithm and reciprocal (about 2 ulp
// each in fp32, far inside the step's error budget); the step kernels use these.
__device__ __forceinline__ float sigmoid_fast(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }
__device__ __forceinline__ float silu_fast(float x) { return __fdividef(x, 1.0f + __expf(-x)); }
__device__ __forceinline__ float softplus_fast(float x)
{
    return fmaxf(x, 0.0f) + __logf(1.0f + __expf(-fabsf(x)));
}
__device__ __forceinline__ float conv4_silu_fast(const float4 w, const float *win, float x)
{
    float acc = w.x * win[0];
    acc = fmaf(w.y, win[1], acc);
    acc = fmaf(w.z, win[2], acc);
    acc = fmaf(w.w, x, acc);
    return silu_fast(acc);
}

__device__ __forceinline__ void store_out4(void *out, size_t idx, int bf16, float a, float b,
                                           float c, float d)
{
    if (bf16) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t *>(&lo);
        pk.y = *reinterpret_cast<uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(out) + idx) = pk;
    } else {
        *reinterpret_cast<float4 *>(reinterpret_cast<float *>(out) + idx) =
            make_float4(a, b, c, d);
    }
}

// ---------------------------------------------------------------- PDL

__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- clusters

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Stores v into the shared-memory word at `local`'s offset inside CTA `rank` of the cluster.
__device__ __forceinline__ void dsmem_store(float *local, uint32_t rank, float v)
{
    uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(a), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

// ---------------------------------------------------------------- mbarrier + TMA bulk copy

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for phase `parity` of `bar` to complete, giving up after about two
// seconds; returns false on time-out (the caller records an error and goes on).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity)
{
    for (uint32_t i = 0; i < 256u; ++i)
        if (mbar_test(bar, parity)) return true;
    for (uint32_t i = 0; i < (1u << 26); ++i) {
        if (mbar_test(bar, parity)) return true;
        __nanosleep(32);
    }
    return false;
}

// Waits for phase `parity` of `bar` with mbarrier.try_wait, which suspends the
// thread in hardware until the phase completes or a short time limit passes, so a
// waiting warp takes no issue slots from the working ones.  Gives up after about
// 2^32 clock cycles (two seconds at 2 GHz) and returns false (the caller records
// an error and goes on).
__device__ __forceinline__ bool mbar_wait_suspend_bounded(uint64_t *bar, uint32_t parity)
{
    const long long t0 = clock64();
    for (;;) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(smem_addr(bar)), "r"(parity)
            : "memory");
        if (ok) return true;
        if (clock64() - t0 > (1LL << 32)) return false;
    }
}

// Waits (acquire at cluster scope) for phase `parity` of a local mbarrier that
// remote CTAs complete with st.async; gives up after about two seconds.
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t *bar, uint32_t parity)
{
    for (uint32_t i = 0; i < (1u << 26); ++i) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(smem_addr(bar)), "r"(parity)
            : "memory");
        if (ok) return true;
        if (i >= 256u) __nanosleep(32);
    }
    return false;
}

// Writes v into the word at `slot`'s offset inside CTA `rank` of the cluster and
// completes 4 bytes of transactions on the mbarrier at `bar`'s offset there.
__device__ __forceinline__ void st_async_remote(float *slot, uint32_t rank, float v, uint64_t *bar)
{
    uint32_t ra, rb;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_addr(slot)), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(smem_addr(bar)), "r"(rank));
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(ra),
                 "r"(__float_as_uint(v)), "r"(rb)
                 : "memory");
}

// One bulk global -> shared copy of `bytes` (multiple of 16, both addresses
// 16-byte aligned) that completes `bytes` transactions on `bar`.
__device__ __forceinline__ void tma_load_1d(void *dst_smem, const void *src_gmem, uint32_t bytes,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// 16 bytes global -> shared without registers (both 16-byte aligned); completes at
// cp_async_wait_all.
__device__ __forceinline__ void cp_async16(void *dst_smem, const void *src_gmem)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst_smem)), "l"(src_gmem)
                 : "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// An L2 policy that marks the lines a load brings in as the first to evict: for data
// read once (weights streamed past the cache), so it does not displace lines that a
// later kernel will read.
__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// tma_load_1d with an L2 cache policy.
__device__ __forceinline__ void tma_load_1d_hint(void *dst_smem, const void *src_gmem, uint32_t bytes,
                                                 uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_addr(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Tiled TMA copies through a tensor map (passed as a __grid_constant__ kernel
// parameter); the innermost coordinate times the element size is a multiple of 16.
__device__ __forceinline__ void tma_load_2d(void *dst_smem, const void *tmap, int x, int y,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_addr(dst_smem)), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y),
        "r"(smem_addr(bar))
        : "memory");
}

// Brings a tensor map (a __grid_constant__ kernel parameter) into the TMA descriptor cache.
__device__ __forceinline__ void prefetch_tensormap(const void *tmap)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *dst_smem, const void *tmap, int x, int y, int z,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(smem_addr(dst_smem)), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z),
        "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(void *dst_smem, const void *tmap, int x, int y, int z, int w,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];"
        ::"r"(smem_addr(dst_smem)), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(w),
        "r"(smem_addr(bar))
        : "memory");
}

}  // namespace dev
}  // namespace gdn
