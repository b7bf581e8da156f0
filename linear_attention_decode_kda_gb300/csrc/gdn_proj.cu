// Projections around the decode step of a KDA layer: the q/k/v rows, the
// low-rank gate chains f = f_b(f_a(x)) and z = g_b(g_a(x)), beta, and the
// output projection.  "Thirty tiny kernels per layer" measures these (not the
// recurrence) as about 90% of a KDA layer's decode time, all of it weight
// streaming; "llama.cpp PR #84" runs f_a beside g_a (and beta) and f_b beside
// g_b as single launches.  Here the q/k/v rows, f_a, g_a and beta share one
// launch (one pass over x), and f_b and g_b another (or, on the column-slab step
// kernel, the step itself: gdn_step.cu).
//
// y[b][n] = sum_k x[b][k] W[n][k]: W is bf16, row-major [N][K], streamed from
// HBM once per pass over the batch rows; x is fp32 or bf16 (a few rows,
// L2-resident); y is fp32.  A launch serves up to four slots, each its own
// (W, x, y).  launch_proj picks one of four kernels by batch rows and K:
//   * proj_tc_kernel (tcgen05, from 16 batch rows);
//   * proj_mma_kernel (warp-level MMA, up to 8 bf16 / 4 fp32 rows shared by the slots);
//   * proj_ring_kernel (CUDA cores, bulk-copy rings, rows of 1024 to 4096);
//   * proj_kernel (CUDA cores, a warp or less per row, the rest).
// Every launch uses programmatic dependent launch, so the next kernel's CTAs start
// beside this one's and the weight stream can begin before the activations exist.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_device.cuh"
#include "gdn_internal.h"
#include "gdn_tc.cuh"
#include "gdn_tmap.h"

namespace gdn {
namespace {

constexpr int PT = 256;  // threads per CTA

struct Slot {
    const __nv_bfloat16 *w;
    const void *x;
    float *y;
    int N, K, ldx, ldy, x_bf16;
    int tpr;   // lanes per row: min(32, K / 8) rounded down to a power of two
    int cta0;  // first CTA of this slot
};

struct Args {
    Slot s[kMaxProjSlots];
    int nslot, B;
    int ksplit;  // tensor-core path: K ranges per output tile (partial sums added atomically)
    int ctas;    // CUDA-core path: CTAs of the launch
    int pf_ctas; // CUDA-core path: the first pf_ctas CTAs ask L2 for every CTA's rows
    int mr_k;    // warp-MMA path: K of every slot
};

__device__ __forceinline__ void unpack8(const uint4 r, float (&v)[8])
{
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}

// Asks L2 for `bytes` (a multiple of 16) from the 16-byte aligned global address p.
__device__ __forceinline__ void prefetch_bulk_l2(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// The weight rows [n0, n0 + nr) of a slot, asked into L2 in pieces of 16 KB spread over
// the lanes of one warp; rows are contiguous, so each piece is one bulk prefetch.
__device__ __forceinline__ void prefetch_rows(const __nv_bfloat16 *w, int K, int n0, int nr, int lane)
{
    if (nr <= 0) return;
    const char *base = reinterpret_cast<const char *>(w + static_cast<size_t>(n0) * K);
    const uint32_t bytes = static_cast<uint32_t>(nr) * static_cast<uint32_t>(K) * 2u;
    for (uint32_t o = static_cast<uint32_t>(lane) * 16384u; o < bytes; o += 32u * 16384u)
        prefetch_bulk_l2(base + o, min(16384u, bytes - o));
}

__device__ __forceinline__ void load_x8(const void *x, size_t idx, int bf16, float (&v)[8])
{
    if (bf16) {
        unpack8(*reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(x) + idx), v);
    } else {
        const float4 a = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(x) + idx);
        const float4 b = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(x) + idx + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
}

// One warp per weight row (half a warp when K is 128 or less), NB batch rows
// accumulated per pass over the row; the sum over the row's lanes is shuffles only.
// Launched with programmatic dependent launch: before the dependency wait the CTA
// only asks L2 for its weight rows (read-only), so the stream of weights overlaps
// the previous kernel; activations are read and outputs written after the wait.
template <int NB>
__global__ void __launch_bounds__(PT) proj_kernel(const __grid_constant__ Args p)
{
    // Before the dependency wait: the first pf_ctas CTAs (those that start early, beside
    // the previous kernel) ask L2 for the rows of CTAs c, c + pf_ctas, ...
    if (threadIdx.x < 32 && static_cast<int>(blockIdx.x) < p.pf_ctas) {
        for (int c = blockIdx.x; c < p.ctas; c += p.pf_ctas) {
            int k = 0;
#pragma unroll
            for (int i = 1; i < kMaxProjSlots; ++i)
                if (i < p.nslot && c >= p.s[i].cta0) k = i;
            const Slot &t = p.s[k];
            const int r = PT / t.tpr, n0 = (c - t.cta0) * r;
            prefetch_rows(t.w, t.K, n0, min(r, t.N - n0), threadIdx.x);
        }
    }
    int si = 0;
#pragma unroll
    for (int k = 1; k < kMaxProjSlots; ++k)
        if (k < p.nslot && static_cast<int>(blockIdx.x) >= p.s[k].cta0) si = k;
    const Slot &s = p.s[si];
    const int tpr = s.tpr, rows = PT / tpr;
    const int r = threadIdx.x / tpr, j = threadIdx.x % tpr;
    const int n = (static_cast<int>(blockIdx.x) - s.cta0) * rows + r;
    const bool valid = n < s.N;
    const int nk = s.K / 8;
    const uint4 *wr = reinterpret_cast<const uint4 *>(s.w + static_cast<size_t>(valid ? n : 0) * s.K);
    dev::pdl_wait();
    // Dependents launch only once this grid has passed its own dependency wait, so a
    // dependent's pre-wait reads overlap this kernel alone, never an earlier one.
    dev::pdl_launch_dependents();

    for (int b0 = 0; b0 < p.B; b0 += NB) {
        float acc[NB];
#pragma unroll
        for (int c = 0; c < NB; ++c) acc[c] = 0.f;
        // U pieces of the row a lane are loaded before any is used (16 for a 4096-wide row
        // measured slower: 128 registers a thread halve the resident warps)
        constexpr int U = 8;
        for (int kb = j; kb < nk; kb += U * tpr) {
            uint4 wv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int kk = kb + u * tpr;
                wv[u] = kk < nk ? __ldg(wr + kk) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int kk = kb + u * tpr;
                if (kk < nk) {
                    float w8[8];
                    unpack8(wv[u], w8);
#pragma unroll
                    for (int c = 0; c < NB; ++c) {
                        if (b0 + c < p.B) {
                            float x8[8];
                            load_x8(s.x, static_cast<size_t>(b0 + c) * s.ldx + kk * 8, s.x_bf16, x8);
#pragma unroll
                            for (int e = 0; e < 8; ++e) acc[c] = fmaf(w8[e], x8[e], acc[c]);
                        }
                    }
                }
            }
        }
        for (int off = tpr >> 1; off > 0; off >>= 1)
#pragma unroll
            for (int c = 0; c < NB; ++c) acc[c] += __shfl_xor_sync(0xffffffffu, acc[c], off);
        if (valid && j == 0) {
#pragma unroll
            for (int c = 0; c < NB; ++c)
                if (b0 + c < p.B) s.y[static_cast<size_t>(b0 + c) * s.ldy + n] = acc[c];
        }
    }
}

__device__ unsigned int g_proj_error;  // bit 0: a bounded mbarrier wait gave up

// ---------------------------------------------------------------- bulk-copy ring
//
// The weight stream for a few batch rows (K <= 4096), by bulk copies: one resident
// CTA an SM, each of its RW warps owning a ring of RING stages of STAGE_B bytes in
// shared memory.  A warp task is a block of contiguous weight rows of one slot that
// fills at most a stage (one row of 4096, or 32 rows of 128); warp w takes tasks
// w, w + W, ... (W warps in all), its lane 0 keeping RING copies in flight, so an SM
// has up to 192 KB of weights on the way.  The first RING copies of every warp are
// issued before the dependency wait (weights are read-only), so a launch queued
// behind another kernel streams its weights into shared memory while that kernel
// runs.  Lanes multiply from shared memory: tpr lanes a row, one 16-byte piece at a
// time, all NB batch rows per piece; the sum over a row's lanes is shuffles only.
constexpr int RW = 8, RING = 3, STAGE_B = 8192;
constexpr int RING_SMEM = RW * RING * STAGE_B;
constexpr int RING_MAX_K = STAGE_B / 2;

template <int NB>
__global__ void __launch_bounds__(RW * 32, 1) proj_ring_kernel(const __grid_constant__ Args p)
{
    extern __shared__ __align__(128) unsigned char rsm[];
    __shared__ __align__(8) uint64_t bar[RW][RING];
    // The slot table in shared memory: indexed by a run-time slot number, the kernel
    // parameter would be read through a generic address on every use.
    __shared__ Slot ss[kMaxProjSlots];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gw = static_cast<int>(blockIdx.x) * RW + warp;
    const int nw = static_cast<int>(gridDim.x) * RW;
    const int ntask = p.ctas, nslot = p.nslot, B = p.B;
    unsigned char *ring = rsm + static_cast<size_t>(warp) * RING * STAGE_B;
    const uint64_t wpol = dev::l2_policy_evict_first();  // weights are read once
#pragma unroll
    for (int i = 0; i < kMaxProjSlots; ++i)
        if (static_cast<int>(threadIdx.x) == i && i < nslot) ss[i] = p.s[i];
    if (lane == 0) {
        for (int i = 0; i < RING; ++i) dev::mbar_init(&bar[warp][i], 1);
        dev::fence_mbar_init();
    }
    __syncthreads();

    // slot, first row and rows of task t
    auto task = [&](int t, int &si, int &n0, int &nr) {
        si = 0;
        for (int k = 1; k < nslot; ++k)
            if (t >= ss[k].cta0) si = k;
        const int K = ss[si].K, rpt = STAGE_B / (2 * K);
        n0 = (t - ss[si].cta0) * rpt;
        nr = min(rpt, ss[si].N - n0);
    };
    auto issue = [&](int k) {  // the warp's k-th task into stage k % RING (lane 0)
        const int t = gw + k * nw;
        if (t >= ntask) return;
        int si, n0, nr;
        task(t, si, n0, nr);
        const int K = ss[si].K;
        const uint32_t bytes = static_cast<uint32_t>(nr) * static_cast<uint32_t>(K) * 2u;
        uint64_t *b = &bar[warp][k % RING];
        dev::mbar_expect_tx(b, bytes);
        dev::tma_load_1d_hint(ring + (k % RING) * STAGE_B, ss[si].w + static_cast<size_t>(n0) * K, bytes, b,
                              wpol);
    };
    if (lane == 0)
        for (int k = 0; k < RING; ++k) issue(k);
    dev::pdl_wait();
    // Dependents launch only once this grid has passed its own dependency wait, so a
    // dependent's pre-wait reads overlap this kernel alone, never an earlier one.
    dev::pdl_launch_dependents();

    bool ok = true;
    for (int k = 0; gw + k * nw < ntask; ++k) {
        const int t = gw + k * nw;
        if (ok) ok = dev::mbar_wait_suspend_bounded(&bar[warp][k % RING], static_cast<uint32_t>((k / RING) & 1));
        int si, n0, nr;
        task(t, si, n0, nr);
        const int K = ss[si].K, tpr = ss[si].tpr, ldx = ss[si].ldx, ldy = ss[si].ldy;
        const bool xb = ss[si].x_bf16 != 0;
        const void *x = ss[si].x;
        float *y = ss[si].y + n0;
        const int rpp = 32 / tpr, nk = K / 8, j = lane % tpr;
        const unsigned char *stage = ring + (k % RING) * STAGE_B;
        for (int r0 = 0; r0 < nr; r0 += rpp) {
            const int r = r0 + lane / tpr;
            float acc[NB];
#pragma unroll
            for (int c = 0; c < NB; ++c) acc[c] = 0.f;
            if (r < nr) {
                const uint4 *wrow = reinterpret_cast<const uint4 *>(stage + static_cast<size_t>(r) * K * 2);
#pragma unroll 4
                for (int kk = j; kk < nk; kk += tpr) {
                    float w8[8];
                    unpack8(wrow[kk], w8);
#pragma unroll
                    for (int c = 0; c < NB; ++c) {
                        if (c < B) {
                            float x8[8];
                            load_x8(x, static_cast<size_t>(c) * ldx + kk * 8, xb, x8);
#pragma unroll
                            for (int e = 0; e < 8; ++e) acc[c] = fmaf(w8[e], x8[e], acc[c]);
                        }
                    }
                }
            }
            for (int off = tpr >> 1; off > 0; off >>= 1)
#pragma unroll
                for (int c = 0; c < NB; ++c) acc[c] += __shfl_xor_sync(0xffffffffu, acc[c], off);
            if (r < nr && j == 0) {
#pragma unroll
                for (int c = 0; c < NB; ++c)
                    if (c < B) y[static_cast<size_t>(c) * ldy + r] = acc[c];
            }
        }
        // the stage is read: the copy of the task RING steps ahead may land there
        dev::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) issue(k + RING);
    }
    if (!ok && lane == 0) {
        // a wait gave up: let every copy still in flight land (bounded) before the CTA
        // releases its shared memory
        int ktot = 0;
        while (gw + ktot * nw < ntask) ++ktot;
        for (int i = 0; i < RING && i < ktot; ++i) {
            const int kl = i + RING * ((ktot - 1 - i) / RING);
            dev::mbar_wait_suspend_bounded(&bar[warp][i], static_cast<uint32_t>((kl / RING) & 1));
        }
        atomicOr(&g_proj_error, 1u);
    }
}

// ---------------------------------------------------------------- warp-MMA GEMV
//
// Up to 8 batch rows of bf16 activations (4 of fp32): the products run on the
// warp-level tensor-core MMA (m16n8k16, bf16 operands, fp32 accumulation).  On CUDA
// cores the weight stream is limited by instructions (each 16-byte piece is unpacked to
// fp32 and multiplied element by element); here one 16-byte load a lane feeds two MMAs.
// A is the activations: batch row g in row g and, with fp32 activations, the bf16
// remainder x - bf16(x) of row g in row g + 8 (each output adds the two rows: about 16
// significant bits of x).  B is eight weight rows: lane (g, j) loads elements
// 8 j ... 8 j + 7 of a 32-column unit of row g and hands them to two MMAs as its
// fragments; the activation fragments follow the same order of k, and a dot product
// does not depend on the order of its terms.
//
// A CTA (16 warps, one an SM) takes tasks of 8 weight rows; its warps split K into
// units of 32 columns and add their partial sums in shared memory in a fixed order.
// Each warp loads a task's weights in one round of 16-byte loads (up to 8 a lane) and
// issues the next task's before it multiplies, so an SM has two tasks in flight; the
// first task's loads go out before the dependency wait (the weights are read-only).
constexpr int MW = 16;                   // warps a CTA
constexpr int MU = 8;                    // 32-column units a warp, at most, per task
constexpr int MMA_MAX_K = MW * MU * 32;  // 4096
constexpr int MXS_MAX = 65536;           // activation fragments in shared memory

__device__ __forceinline__ uint4 ldg_stream(const void *ptr, uint64_t policy)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(ptr), "l"(policy));
    return v;
}

// d += A (16 x 16 bf16, row fragments a) * B (16 x 8 bf16, column fragments b0 b1)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                 "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// bf16 pair (u, v) and the pair of remainders (u - bf16(u), v - bf16(v)), the first
// element in the low half
__device__ __forceinline__ void split_pair(float u, float v, uint32_t &hi, uint32_t &lo)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(u, v);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(u - hf.x, v - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

template <bool SPLIT>
__global__ void __launch_bounds__(MW * 32, 1) proj_mma_kernel(const __grid_constant__ Args p)
{
    extern __shared__ __align__(16) unsigned char msm[];  // activation fragments
    __shared__ Slot ss[kMaxProjSlots];
    __shared__ float red[2][MW][64];  // a warp's partial outputs: batch row g, task row n at 8 g + n
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, j = lane & 3;
    const int ntile = p.ctas, nslot = p.nslot, B = p.B, K = p.mr_k, nl = 4 * B;
    const int nu = K / 32, u0 = warp * nu / MW, u1 = (warp + 1) * nu / MW;  // this warp's units
    const uint64_t pol = dev::l2_policy_evict_first();  // weights are read once
#pragma unroll
    for (int i = 0; i < kMaxProjSlots; ++i)
        if (static_cast<int>(threadIdx.x) == i && i < nslot) ss[i] = p.s[i];
    __syncthreads();

    // slot, first row and rows of task t
    auto task = [&](int t, int &si, int &r0, int &nr) {
        si = 0;
        for (int k = 1; k < nslot; ++k)
            if (t >= ss[k].cta0) si = k;
        r0 = (t - ss[si].cta0) * 8;
        nr = min(8, ss[si].N - r0);
    };
    // this lane's weights of task t: row r0 + g, elements 8 j ... 8 j + 7 of each unit
    auto load = [&](int t, uint4 (&w)[MU]) {
        int si, r0, nr;
        task(t, si, r0, nr);
        const __nv_bfloat16 *row = ss[si].w + static_cast<size_t>(r0 + (g < nr ? g : 0)) * K + j * 8;
#pragma unroll
        for (int u = 0; u < MU; ++u)
            w[u] = (u0 + u < u1 && g < nr) ? ldg_stream(row + (u0 + u) * 32, pol) : make_uint4(0u, 0u, 0u, 0u);
    };

    uint4 wa[MU], wb[MU];
    int t = blockIdx.x;
    load(t, wa);
    dev::pdl_wait();
    // Dependents launch only once this grid has passed its own dependency wait, so a
    // dependent's pre-wait reads overlap this kernel alone, never an earlier one.
    dev::pdl_launch_dependents();

    // Activation fragments, unit major: entry (u, l) for lane l < 4B holds row g = l / 4,
    // elements 32 u + 8 (l % 4) ... + 7 (fp32 activations: the bf16 pairs, then their
    // remainders).
    uint4 *xs4 = reinterpret_cast<uint4 *>(msm);
    {
        const void *x = ss[0].x;
        const int ldx = ss[0].ldx;
        for (int i = threadIdx.x; i < nu * nl; i += MW * 32) {
            const int u = i / nl, l = i - u * nl;
            const size_t off = static_cast<size_t>(l >> 2) * ldx + u * 32 + (l & 3) * 8;
            if (SPLIT) {
                const float4 e0 = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(x) + off);
                const float4 e1 = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(x) + off + 4);
                uint4 hi, lo;
                split_pair(e0.x, e0.y, hi.x, lo.x);
                split_pair(e0.z, e0.w, hi.y, lo.y);
                split_pair(e1.x, e1.y, hi.z, lo.z);
                split_pair(e1.z, e1.w, hi.w, lo.w);
                xs4[2 * i] = hi;
                xs4[2 * i + 1] = lo;
            } else {
                xs4[i] = *reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(x) + off);
            }
        }
    }
    __syncthreads();

    for (int par = 0; t < ntile; t += gridDim.x, par ^= 1) {
        if (t + static_cast<int>(gridDim.x) < ntile) load(t + gridDim.x, wb);  // in flight meanwhile
        float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int u = 0; u < MU; ++u) {
            if (u0 + u < u1) {
                uint32_t a[4] = {0u, 0u, 0u, 0u}, c[4] = {0u, 0u, 0u, 0u};
                if (lane < nl) {
                    const int e = (u0 + u) * nl + lane;
                    if (SPLIT) {
                        const uint4 hi = xs4[2 * e], lo = xs4[2 * e + 1];
                        a[0] = hi.x; a[1] = lo.x; a[2] = hi.y; a[3] = lo.y;
                        c[0] = hi.z; c[1] = lo.z; c[2] = hi.w; c[3] = lo.w;
                    } else {
                        const uint4 v = xs4[e];
                        a[0] = v.x; a[2] = v.y;
                        c[0] = v.z; c[2] = v.w;
                    }
                }
                mma_bf16_16816(d[0], a, wa[u].x, wa[u].y);
                mma_bf16_16816(d[1], c, wa[u].z, wa[u].w);
            }
        }
        // lane (g, j): batch row g, task rows 2 j and 2 j + 1 (MMA rows g + 8 carry the
        // remainders' share, zero for bf16 activations)
        if (g < B) {
            red[par][warp][g * 8 + 2 * j] = (d[0][0] + d[1][0]) + (d[0][2] + d[1][2]);
            red[par][warp][g * 8 + 2 * j + 1] = (d[0][1] + d[1][1]) + (d[0][3] + d[1][3]);
        }
        __syncthreads();
        if (static_cast<int>(threadIdx.x) < 8 * B) {
            int si, r0, nr;
            task(t, si, r0, nr);
            const int gb = threadIdx.x >> 3, n = threadIdx.x & 7;
            if (n < nr) {
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < MW; ++w) v += red[par][w][gb * 8 + n];
                ss[si].y[static_cast<size_t>(gb) * ss[si].ldy + r0 + n] = v;
            }
        }
#pragma unroll
        for (int u = 0; u < MU; ++u) wa[u] = wb[u];
    }
}

// ---------------------------------------------------------------- tcgen05 path
//
// From 16 batch rows up the products are dense enough for the tensor core: a
// CTA takes 128 weight rows (M) against up to 64 batch rows (N), K in tiles of
// 64 through a ring of shared-memory stages fed by TMA.  Activations are bf16
// (the layer input) or fp32 rows split into bf16 hi + lo, multiplied as W hi +
// W lo (the weights are exact in bf16).  The fp32 accumulator lives in TMEM.

constexpr int TC_M = 128, TC_N = 64, TC_K = 64, TC_PT = 128;
constexpr int TC_WB = TC_M * TC_K * 2;   // weight tile bytes
constexpr int TC_XB = TC_N * TC_K * 2;   // bf16 activation tile (or one half of the split)
// A weight tile arrives by one TMA box of 64 elements x 128 rows in the 128-byte
// swizzled K-major layout (tc::op_desc_sw128).  Activation rows arrive as a plain
// [64][64] box and the threads copy them into the canonical layout (tc::op_offset):
// bf16 as is, fp32 split into bf16 hi and lo.
template <bool SPLIT> struct TcCfg {
    static constexpr int RAW = TC_WB + (SPLIT ? 2 : 1) * TC_XB;  // the activation box
    static constexpr int RAW_BYTES = TC_N * TC_K * (SPLIT ? 4 : 2);
    static constexpr int STAGE = RAW + RAW_BYTES;
    static constexpr int NS = SPLIT ? 4 : 6;  // one CTA an SM
    static constexpr int LAG = 2;             // refills reuse the stage of the tile 2 back
    // CTAs to aim for when splitting K (the split's zeroing memsets cost about as much
    // as a second wave, so a launch that already covers most SMs stays unsplit)
    static constexpr int TARGET = 160;
    static constexpr int D = NS - LAG;   // tiles in flight ahead of the product
    static constexpr int SMEM = NS * STAGE;
    static constexpr uint32_t TX = TC_WB + RAW_BYTES;
};

struct TcMaps {
    CUtensorMap w[kMaxProjSlots], x[kMaxProjSlots];
};


// Launches with programmatic dependent launch: the kernels wait for the previous
// kernel on the stream before they read activations or write outputs.
template <typename... KArgs, typename... Args2>
cudaError_t launch_pdl(void (*fn)(KArgs...), dim3 grid, int threads, int smem, cudaStream_t stream,
                       Args2... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, args...);
}

// SMs of the current device (cached per device).
int num_sms()
{
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
        cache[dev] = n;
    }
    return cache[dev];
}

struct TcShared {
    uint64_t full[8];  // the tile of stage s has arrived
    uint64_t done[8];  // the products that read stage s have completed
    uint32_t tmem;
};

template <bool SPLIT>
__global__ void __launch_bounds__(TC_PT, 1)
proj_tc_kernel(const __grid_constant__ Args p, const __grid_constant__ TcMaps maps)
{
    using Cfg = TcCfg<SPLIT>;
    constexpr int NS = Cfg::NS, STAGE = Cfg::STAGE, D = Cfg::D;
    extern __shared__ __align__(1024) unsigned char sm[];
    __shared__ __align__(16) TcShared ts;
    int si = 0;
#pragma unroll
    for (int k = 1; k < kMaxProjSlots; ++k)
        if (k < p.nslot && static_cast<int>(blockIdx.x) >= p.s[k].cta0) si = k;
    const Slot &s = p.s[si];
    const CUtensorMap *mw = &maps.w[si], *mx = &maps.x[si];
    const int tid = threadIdx.x, warp = tid >> 5;
    const int n0 = (static_cast<int>(blockIdx.x) - s.cta0) * TC_M;  // first weight row
    const int b0 = blockIdx.y * TC_N;                                // first batch row
    const int nb = min(TC_N, p.B - b0);
    const int nk = s.K / TC_K / p.ksplit;                           // K tiles of this CTA
    const int kt0 = blockIdx.z * nk;                                 // its first K tile

    if (warp == 0) tc::tmem_alloc(&ts.tmem, TC_N);
    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            dev::mbar_init(&ts.full[i], 1);
            dev::mbar_init(&ts.done[i], 1);
        }
        dev::fence_mbar_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = ts.tmem;

    // tile kt into stage kt % NS (rows past N or past the batch read as zero)
    auto load = [&](int kt) {
        unsigned char *st = sm + (kt % NS) * STAGE;
        dev::mbar_expect_tx(&ts.full[kt % NS], Cfg::TX);
        dev::tma_load_2d(st, mw, (kt0 + kt) * TC_K, n0, &ts.full[kt % NS]);
        dev::tma_load_2d(st + Cfg::RAW, mx, (kt0 + kt) * TC_K, b0, &ts.full[kt % NS]);
    };

    bool ok = true;
    const uint32_t idesc = tc::idesc_f16(TC_M, TC_N, false, true);
    // Asking L2 for the weights before the wait measured slower here (B64 layer: 150.8
    // against 146.7 us): the TMA ring already keeps the weight stream busy.
    dev::pdl_wait();
    // Dependents launch only once this grid has passed its own dependency wait, so a
    // dependent's pre-wait reads overlap this kernel alone, never an earlier one.
    dev::pdl_launch_dependents();
    if (tid == 0) {
        dev::prefetch_tensormap(mw);
        dev::prefetch_tensormap(mx);
        for (int kt = 0; kt < D && kt < nk; ++kt) load(kt);
    }
#pragma unroll 1
    for (int kt = 0; kt < nk; ++kt) {
        unsigned char *st = sm + (kt % NS) * STAGE;
        if (ok) ok = dev::mbar_wait_bounded(&ts.full[kt % NS], static_cast<uint32_t>((kt / NS) & 1));
        // the activation box -> the canonical layout: fp32 as bf16 hi and lo, bf16 as is
        if (SPLIT) {
            const float *xf = reinterpret_cast<const float *>(st + Cfg::RAW);
#pragma unroll
            for (int e = 0; e < TC_N * 16 / TC_PT; ++e) {
                const int pc = tid + e * TC_PT, r = pc >> 4, q = pc & 15;
                const float4 v = *reinterpret_cast<const float4 *>(xf + r * TC_K + 4 * q);
                const __nv_bfloat162 h0 = __floats2bfloat162_rn(v.x, v.y), h1 = __floats2bfloat162_rn(v.z, v.w);
                const float2 f0 = __bfloat1622float2(h0), f1 = __bfloat1622float2(h1);
                const __nv_bfloat162 l0 = __floats2bfloat162_rn(v.x - f0.x, v.y - f0.y);
                const __nv_bfloat162 l1 = __floats2bfloat162_rn(v.z - f1.x, v.w - f1.y);
                unsigned char *hi = st + TC_WB + tc::op_offset(r, 4 * q, TC_K);
                uint2 hv, lv;
                hv.x = *reinterpret_cast<const uint32_t *>(&h0);
                hv.y = *reinterpret_cast<const uint32_t *>(&h1);
                lv.x = *reinterpret_cast<const uint32_t *>(&l0);
                lv.y = *reinterpret_cast<const uint32_t *>(&l1);
                *reinterpret_cast<uint2 *>(hi) = hv;
                *reinterpret_cast<uint2 *>(hi + TC_XB) = lv;
            }
        } else {
            const unsigned char *xb = st + Cfg::RAW;
#pragma unroll
            for (int e = 0; e < TC_N * 8 / TC_PT; ++e) {
                const int pc = tid + e * TC_PT, r = pc >> 3, q = pc & 7;
                *reinterpret_cast<uint4 *>(st + TC_WB + tc::op_offset(r, 8 * q, TC_K)) =
                    *reinterpret_cast<const uint4 *>(xb + (r * TC_K + 8 * q) * 2);
            }
        }
        dev::fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after_sync();
            const uint32_t sa = tc::smem_u32(st);
#pragma unroll
            for (int ks = 0; ks < TC_K; ks += 16) {
                const uint64_t dw = tc::op_desc_sw128(sa, ks);
                tc::mma_f16(tm, dw, tc::op_desc(sa + TC_WB, ks, TC_K), idesc, kt > 0 || ks > 0);
                if (SPLIT) tc::mma_f16(tm, dw, tc::op_desc(sa + TC_WB + TC_XB, ks, TC_K), idesc, true);
            }
            tc::mma_commit(&ts.done[kt % NS]);
            // tile kt + D goes where tile kt + D - NS (= kt - LAG) was, once its products are done
            const int kn = kt + D;
            if (kn < nk) {
                if (kn >= NS && ok)
                    ok = dev::mbar_wait_bounded(&ts.done[kn % NS], static_cast<uint32_t>(((kn - NS) / NS) & 1));
                load(kn);
            }
        }
    }
    // the last tile's products, then the accumulator out: lane = weight row
    if (nk > 0 && ok)
        ok = dev::mbar_wait_bounded(&ts.done[(nk - 1) % NS], static_cast<uint32_t>(((nk - 1) / NS) & 1));
    tc::fence_after_sync();
    const int n = n0 + tid;
#pragma unroll
    for (int c0 = 0; c0 < TC_N; c0 += 16) {
        float v[16];
        tc::tmem_ld16(tc::taddr(tm, 32 * warp, c0), v);
        if (n < s.N)
#pragma unroll
            for (int c = 0; c < 16; ++c)
                if (c0 + c < nb) {
                    float *yp = s.y + static_cast<size_t>(b0 + c0 + c) * s.ldy + n;
                    if (p.ksplit > 1)
                        atomicAdd(yp, v[c]);
                    else
                        *yp = v[c];
                }
    }
    if (!ok) {
        // a wait gave up: let every copy and product land (bounded) before the
        // shared memory and TMEM are released
        if (tid == 0) {
            for (int i = 0; i < NS && i < nk; ++i) {
                const int last = i + NS * ((nk - 1 - i) / NS);
                dev::mbar_wait_bounded(&ts.full[i], static_cast<uint32_t>((last / NS) & 1));
                dev::mbar_wait_bounded(&ts.done[i], static_cast<uint32_t>((last / NS) & 1));
            }
            atomicOr(&g_proj_error, 1u);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, TC_N);
}

template <bool SPLIT>
cudaError_t launch_tc(const Args &a, const ProjSlotDesc *slots, int ctas, int B, cudaStream_t stream)
{
    static bool attr_set[64];  // per device; benign race: every writer sets the same value
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(proj_tc_kernel<SPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 TcCfg<SPLIT>::SMEM);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    TcMaps m = {};
    for (int i = 0; i < a.nslot; ++i) {
        const ProjSlotDesc &d = slots[i];
        {   // weights [N][K]: boxes of 64 elements x 128 rows, 128-byte swizzled
            const uint64_t dim[2] = {static_cast<uint64_t>(d.K), static_cast<uint64_t>(d.N)};
            const uint64_t stride[1] = {static_cast<uint64_t>(d.K) * 2};
            const uint32_t box[2] = {TC_K, TC_M};
            if (!encode_tiled_swizzled(&m.w[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d.w, dim, stride, box,
                                       CU_TENSOR_MAP_SWIZZLE_128B))
                return cudaErrorInvalidValue;
        }
        {   // activation rows [B][ldx] as a [B][K] box of 64 rows x 64
            const uint64_t dim[2] = {static_cast<uint64_t>(d.K), static_cast<uint64_t>(B)};
            const uint64_t stride[1] = {static_cast<uint64_t>(d.ldx) * (SPLIT ? 4 : 2)};
            const uint32_t box[2] = {TC_K, TC_N};
            if (!encode_tiled(&m.x[i], SPLIT ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                              2, d.x, dim, stride, box))
                return cudaErrorInvalidValue;
        }
    }
    if (a.ksplit > 1)  // partial sums are added into zeroed outputs
        for (int i = 0; i < a.nslot; ++i) {
            e = cudaMemset2DAsync(slots[i].y, static_cast<size_t>(slots[i].ldy) * sizeof(float), 0,
                                  static_cast<size_t>(slots[i].N) * sizeof(float), B, stream);
            if (e != cudaSuccess) return e;
        }
    return launch_pdl(proj_tc_kernel<SPLIT>, dim3(ctas, (B + TC_N - 1) / TC_N, a.ksplit), TC_PT,
                      TcCfg<SPLIT>::SMEM, stream, a, m);
}

}  // namespace

bool proj_slot_ok(const ProjSlotDesc &d)
{
    const auto al16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
    const int es = d.x_bf16 ? 2 : 4;
    return d.w && d.x && d.y && d.N > 0 && d.K >= 8 && d.K % 8 == 0 && al16(d.w) && al16(d.x) &&
           (static_cast<long long>(d.ldx) * es) % 16 == 0 && d.ldx >= d.K && d.ldy >= d.N &&
           (reinterpret_cast<uintptr_t>(d.y) & 3u) == 0;
}

cudaError_t launch_proj(const ProjSlotDesc *slots, int nslot, int B, cudaStream_t stream, bool prefetch)
{
    if (nslot < 1 || nslot > kMaxProjSlots || B < 0) return cudaErrorInvalidValue;
    if (B == 0) return cudaSuccess;
    Args a = {};
    a.nslot = nslot;
    a.B = B;
    a.ksplit = 1;
    int ctas = 0;
    for (int i = 0; i < nslot; ++i) {
        const ProjSlotDesc &d = slots[i];
        if (!proj_slot_ok(d)) return cudaErrorInvalidValue;
        int tpr = 1;  // lanes per row: up to a warp, one 16-byte piece of K each
        while (tpr < 32 && tpr * 2 <= d.K / 8) tpr *= 2;
        Slot &s = a.s[i];
        s.w = static_cast<const __nv_bfloat16 *>(d.w);
        s.x = d.x;
        s.y = d.y;
        s.N = d.N;
        s.K = d.K;
        s.ldx = d.ldx;
        s.ldy = d.ldy;
        s.x_bf16 = d.x_bf16;
        s.tpr = tpr;
        s.cta0 = ctas;
        const int rows = PT / tpr;
        ctas += (d.N + rows - 1) / rows;
    }
    // tcgen05 from kProjTcMinBatch batch rows, when every slot's K is a multiple of
    // 64 and all slots read activations of one type
    bool tc_ok = B >= kProjTcMinBatch;
    for (int i = 0; i < nslot; ++i)
        tc_ok = tc_ok && slots[i].K % TC_K == 0 && slots[i].N % 8 == 0 &&
                slots[i].x_bf16 == slots[0].x_bf16;
    if (tc_ok) {
        int tctas = 0, kmin = 1 << 30;
        for (int i = 0; i < nslot; ++i) {
            a.s[i].cta0 = tctas;
            tctas += (slots[i].N + TC_M - 1) / TC_M;
            kmin = min(kmin, slots[i].K / TC_K);
        }
        // split K until the launch covers the SMs (every slot's K tiles divide evenly)
        const int ctas_y = tctas * ((B + TC_N - 1) / TC_N);
        a.ksplit = 1;
        const int target = slots[0].x_bf16 ? TcCfg<false>::TARGET : TcCfg<true>::TARGET;
        while (ctas_y * a.ksplit * 2 <= target && a.ksplit * 2 <= kmin) {
            bool even = true;
            for (int i = 0; i < nslot; ++i) even = even && (slots[i].K / TC_K) % (a.ksplit * 2) == 0;
            if (!even) break;
            a.ksplit *= 2;
        }
        return slots[0].x_bf16 ? launch_tc<false>(a, slots, tctas, B, stream)
                               : launch_tc<true>(a, slots, tctas, B, stream);
    }
    // the warp-MMA GEMV: every slot reads the same activations (up to 8 bf16 rows, 4
    // fp32) against K columns, a multiple of 32 up to 4096
    bool mma_ok = B <= (slots[0].x_bf16 ? 8 : 4) && slots[0].K % 32 == 0 && slots[0].K <= MMA_MAX_K;
    for (int i = 1; i < nslot; ++i)
        mma_ok = mma_ok && slots[i].K == slots[0].K && slots[i].x == slots[0].x &&
                 slots[i].ldx == slots[0].ldx && slots[i].x_bf16 == slots[0].x_bf16;
    const int xs_bytes = B * slots[0].K * (slots[0].x_bf16 ? 2 : 4);
    if (mma_ok && xs_bytes <= MXS_MAX) {
        static bool mma_attr[64];  // per device; benign race: every writer sets the same value
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        if (!mma_attr[dev]) {
            for (void (*f)(Args) : {proj_mma_kernel<false>, proj_mma_kernel<true>}) {
                e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, MXS_MAX);
                if (e != cudaSuccess) return e;
            }
            mma_attr[dev] = true;
        }
        int tasks = 0;
        for (int i = 0; i < nslot; ++i) {
            a.s[i].cta0 = tasks;
            tasks += (slots[i].N + 7) / 8;
        }
        a.ctas = tasks;
        a.mr_k = slots[0].K;
        return launch_pdl(slots[0].x_bf16 ? proj_mma_kernel<false> : proj_mma_kernel<true>,
                          dim3(max(1, min(num_sms(), tasks))), MW * 32, xs_bytes, stream, a);
    }
    int kmax = 0;
    for (int i = 0; i < nslot; ++i) kmax = max(kmax, slots[i].K);
    // narrow rows (the low-rank gate pair, K = rank) stay on the per-row kernel below,
    // which spreads them over more warps
    if (kmax >= 1024 && kmax <= RING_MAX_K && B <= 16) {
        // the bulk-copy ring (every batch row in one pass over the weights): tasks of
        // STAGE_B / (2 K) rows, one resident CTA an SM
        static bool ring_attr[64];  // per device; benign race: every writer sets the same value
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        if (!ring_attr[dev]) {
            for (void (*f)(Args) : {proj_ring_kernel<1>, proj_ring_kernel<2>, proj_ring_kernel<4>,
                                    proj_ring_kernel<8>, proj_ring_kernel<16>}) {
                e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, RING_SMEM);
                if (e != cudaSuccess) return e;
            }
            ring_attr[dev] = true;
        }
        int tasks = 0;
        for (int i = 0; i < nslot; ++i) {
            a.s[i].cta0 = tasks;
            const int rpt = STAGE_B / (2 * slots[i].K);
            tasks += (slots[i].N + rpt - 1) / rpt;
        }
        a.ctas = tasks;
        void (*fn)(Args) = B > 8 ? proj_ring_kernel<16> : B > 4 ? proj_ring_kernel<8>
                         : B > 2 ? proj_ring_kernel<4> : B > 1 ? proj_ring_kernel<2> : proj_ring_kernel<1>;
        return launch_pdl(fn, dim3(max(1, min(num_sms(), (tasks + RW - 1) / RW))), RW * 32, RING_SMEM,
                          stream, a);
    }
    a.ctas = ctas;
    a.pf_ctas = prefetch ? min(ctas, num_sms()) : 0;
    void (*fn)(Args) = B >= 8 ? proj_kernel<8> : B >= 4 ? proj_kernel<4> : B >= 2 ? proj_kernel<2>
                                                                           : proj_kernel<1>;
    return launch_pdl(fn, dim3(ctas), PT, 0, stream, a);
}

}  // namespace gdn

namespace gdn {

unsigned int take_proj_error()
{
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_proj_error, sizeof(v)) != cudaSuccess) return ~0u;
    if (v && cudaMemcpyToSymbol(g_proj_error, &zero, sizeof(zero)) != cudaSuccess) return ~0u;
    return v;
}

}  // namespace gdn
