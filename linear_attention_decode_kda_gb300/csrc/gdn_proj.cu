// Projections around the decode step of a KDA layer: the q/k/v rows, the
// low-rank gate chains f = f_b(f_a(x)) and z = g_b(g_a(x)), beta, and the
// output projection.  "Thirty tiny kernels per layer" measures these (not the
// recurrence) as about 90% of a KDA layer's decode time, all of it weight
// streaming; "llama.cpp PR #84" runs f_a beside g_a (and beta) and f_b beside
// g_b as single launches.  Here the q/k/v rows, f_a, g_a and beta share one
// launch (one pass over x), and f_b and g_b another.
//
// y[b][n] = sum_k x[b][k] W[n][k]: W is bf16, row-major [N][K], streamed from
// HBM once per 8 batch rows; x is fp32 or bf16 (a few rows, L2-resident); y is
// fp32.  A launch serves up to four slots, each its own (W, x, y); the grid
// covers all rows of all slots, a warp (or less) per row reading K in 16-byte pieces.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_internal.h"

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
template <int NB>
__global__ void __launch_bounds__(PT) proj_kernel(const __grid_constant__ Args p)
{
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

    for (int b0 = 0; b0 < p.B; b0 += NB) {
        float acc[NB];
#pragma unroll
        for (int c = 0; c < NB; ++c) acc[c] = 0.f;
#pragma unroll 8
        for (int kk = j; kk < nk; kk += tpr) {
            float w8[8];
            unpack8(__ldg(wr + kk), w8);
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

}  // namespace

bool proj_slot_ok(const ProjSlotDesc &d)
{
    const auto al16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
    const int es = d.x_bf16 ? 2 : 4;
    return d.w && d.x && d.y && d.N > 0 && d.K >= 8 && d.K % 8 == 0 && al16(d.w) && al16(d.x) &&
           (static_cast<long long>(d.ldx) * es) % 16 == 0 && d.ldx >= d.K && d.ldy >= d.N &&
           (reinterpret_cast<uintptr_t>(d.y) & 3u) == 0;
}

cudaError_t launch_proj(const ProjSlotDesc *slots, int nslot, int B, cudaStream_t stream)
{
    if (nslot < 1 || nslot > kMaxProjSlots || B < 0) return cudaErrorInvalidValue;
    if (B == 0) return cudaSuccess;
    Args a = {};
    a.nslot = nslot;
    a.B = B;
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
    if (B >= 8)
        proj_kernel<8><<<ctas, PT, 0, stream>>>(a);
    else if (B >= 4)
        proj_kernel<4><<<ctas, PT, 0, stream>>>(a);
    else if (B >= 2)
        proj_kernel<2><<<ctas, PT, 0, stream>>>(a);
    else
        proj_kernel<1><<<ctas, PT, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace gdn
