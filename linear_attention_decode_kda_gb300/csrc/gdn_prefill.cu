// Prefill of T tokens per sequence; state and conv window advanced in place.
//
// Gated DeltaNet (one decay per head), d_k = d_v = 128, bf16 inputs: the
// chunked WY/UT form ("llama.cpp PR #84", chunked KDA prefill; the gate here
// is per head) on tcgen05 tensor cores.  Other shapes run the T tokens
// through the recurrent step kernel.
//
// Per chunk of C = 32 tokens with start state S0 (G_t = cumulative log-decay
// inside the chunk, every exponent <= 0):
//   A[t][s] = beta_t (k_t . k_s) e^{G_t - G_s}   (s < t),   T = (I + A)^-1
//   W = T (beta e^G k),  U = T (beta v),  V_new = U - W S0
//   O = (e^G q) S0 + M V_new,   M[t][s] = (q_t . k_s) e^{G_t - G_s}  (s <= t)
//   S = e^{G_last} S0 + (k e^{G_last - G})^T V_new
// Operands are fp16 (kind::f16), accumulation fp32.
// Everything is computed transposed so that every product has M = 128 rows
// (the head dimension) on the tensor core: S^T (d_v x d_k, fp32) lives in TMEM
// as an accumulator, V_new^T, O^T, W^T, U^T too.  The q/k L2 norms come from
// the diagonal of one Gram product [k; q] [k; q]^T whose off-diagonal blocks
// give k.k and q.k.  The triangular inverse is a blocked forward substitution
// in fp32 on the CUDA cores.  One CTA (8 warps) owns one (sequence, value
// head); value heads sharing a qk head form a thread-block cluster so the
// shared q/k conv rows are written only after every CTA has read them.
#include "gdn_device.cuh"
#include "gdn_prefill.h"
#include "gdn_tc.cuh"
#include "gdn_tmap.h"

#include <cuda.h>
#include <cuda_fp16.h>

namespace gdn {
namespace {

using namespace dev;

constexpr int PD = 128;   // d_k = d_v
constexpr int CH = 32;    // chunk length
constexpr int PT = 256;   // threads: warps w and w + 4 share TMEM lane quadrant w and split columns
constexpr int KM1 = 3;

// Dynamic shared memory (bytes).  Regions are reused once their readers are done.
// Operands marked "split" are stored as fp16 hi and lo halves (x ~ hi + lo).
constexpr int SM_RAW = 0;                          // [3][CH][PD] bf16 q, k, v rows of the chunk
constexpr int SM_Z = SM_RAW + CH * 3 * PD * 2;     // [CH][PD] bf16 output-gate rows
constexpr int SM_ST = SM_Z + CH * PD * 2;          // split S^T [PD x PD]: hi, then lo
constexpr int SM_R1 = SM_ST + 2 * PD * PD * 2;     // [k; q] hi over [k; q] lo as one 128-row
                                                   // operand -> W [CH x PD] -> o^2 [PD][CH] f32
constexpr int SM_R2 = SM_R1 + 2 * 2 * CH * PD * 2; // split (beta v)^T, k_bg^T -> split V_new^T, M
constexpr int SM_R3 = SM_R2 + 3 * PD * CH * 2;     // split (e^G q), split k_t^T
constexpr int SM_R4 = SM_R3 + 4 * CH * PD * 2;     // T [CH x CH]
constexpr int SM_R5 = SM_R4 + CH * CH * 2;         // Gram f32 [2CH][2CH], A f32, T f32
constexpr int GS = 2 * CH + 1;                     // padded row stride of the f32 Gram
constexpr int SQS = PD + 1;                         // padded row stride of the o^2 scratch
constexpr int YS = PD + 4;                          // row stride of the y staging rows (16-byte aligned)
constexpr int SM_BYTES = SM_R5 + 2 * CH * GS * 4 + 2 * CH * CH * 4;
// operand offsets inside the regions
constexpr int OP_VB = 0, OP_KBG = 2 * PD * CH * 2;                  // R2 (first use)
constexpr int OP_VN = 0, OP_M = 2 * PD * CH * 2;                    // R2 (second use)
constexpr int OP_QG = 0, OP_KT = 2 * CH * PD * 2;                   // R3
constexpr int F_GRAM = 0, F_A = 2 * CH * GS * 4, F_T = F_A + CH * CH * 4;  // R5 (bytes)

// TMEM columns.
constexpr int TM_GRAM = 0;    // 128 columns: [k; q]_{hi;lo} [k; q]_{hi;lo}^T
constexpr int TM_WT = 128;    // CH: W^T
constexpr int TM_UT = 160;    // CH: U^T, then V_new^T
constexpr int TM_OT = 192;    // CH: O^T
constexpr int TM_ST = 256;    // 128: S^T

__device__ unsigned int g_prefill_error;  // bit 0: a bounded mbarrier wait gave up

struct PrefillShared {
    float G[CH], eG[CH], beta[CH], rk[CH], rq[CH], rinv[CH];
    float Rt[16][16];
    uint64_t raw_full, z_full, mma_bar;
    uint32_t tmem;
};

// Tensor-core operands are fp16 (11 significant bits); the precision-critical
// ones are kept as hi + lo pairs and multiplied as hi*hi + hi*lo + lo*hi.
__device__ __forceinline__ void put_h(unsigned char *base, uint32_t off, float v)
{
    *reinterpret_cast<__half *>(base + off) = __float2half_rn(v);
}
using tc::mma_chain;
using tc::mma_split;
using tc::put_row8;
using tc::put_split;
__device__ __forceinline__ float get_h(const unsigned char *base, uint32_t off)
{
    return __half2float(*reinterpret_cast<const __half *>(base + off));
}
__device__ __forceinline__ float get_bf16(const unsigned char *base, uint32_t off)
{
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(base + off));
}

// SiLU with the hardware exponential and fast division (relative error ~1e-6,
// far below the tensor-core operand rounding of this path).
__device__ __forceinline__ float silu_fast(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

__device__ __forceinline__ float conv4_silu_fast(const float4 w, const float *win, float x)
{
    float acc = w.x * win[0];
    acc = fmaf(w.y, win[1], acc);
    acc = fmaf(w.z, win[2], acc);
    acc = fmaf(w.w, x, acc);
    return silu_fast(acc);
}

// Makes this thread's shared-memory writes visible to the tensor core, then syncs the CTA.
__device__ __forceinline__ void publish_smem()
{
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
}

__global__ void __launch_bounds__(PT, 1)
chunk_prefill_kernel(const StepArgs a, const __grid_constant__ CUtensorMap tm_qkv,
                     const __grid_constant__ CUtensorMap tm_z)
{
    extern __shared__ __align__(1024) unsigned char sm[];
    __shared__ __align__(16) PrefillShared ps;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, half = warp >> 2;
    const int ch = tid & (PD - 1);  // channel / TMEM lane of this thread
    const int lb = 32 * quad;       // this warp's TMEM lane quadrant
    const int h = blockIdx.x, b = blockIdx.y, hq = h / a.group;
    const int T = a.T, Ts = a.Ts, C = a.C, H = a.H_v;
    const bool clustered = a.group > 1;
    const bool qk_owner = (h % a.group) == 0;
    const size_t head = static_cast<size_t>(b) * H + h;
    unsigned char *raw = sm + SM_RAW, *zs = sm + SM_Z;
    unsigned char *st_hi = sm + SM_ST, *st_lo = sm + SM_ST + PD * PD * 2;
    unsigned char *r1 = sm + SM_R1, *r2 = sm + SM_R2, *r3 = sm + SM_R3, *r4 = sm + SM_R4;
    float *Gf = reinterpret_cast<float *>(sm + SM_R5 + F_GRAM);   // [2CH][GS]
    float *Af = reinterpret_cast<float *>(sm + SM_R5 + F_A);      // [CH][CH]
    float *Tf = reinterpret_cast<float *>(sm + SM_R5 + F_T);      // [CH][CH]
    const int chq = hq * PD, chk = a.H_qk * PD + hq * PD, chv = 2 * a.H_qk * PD + h * PD;
    constexpr int NR = 2 * CH;  // rows of [k; q]; the lo copy follows as rows NR .. 2NR-1

    if (warp == 0) tc::tmem_alloc(&ps.tmem, 512);
    if (tid == 0) {
        mbar_init(&ps.raw_full, 1);
        mbar_init(&ps.z_full, 1);
        mbar_init(&ps.mma_bar, 1);
        fence_mbar_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = ps.tmem;
    pdl_wait();
    // Dependents launch only once this grid has passed its own dependency wait, so a
    // dependent's pre-wait reads overlap this kernel alone, never an earlier one.
    pdl_launch_dependents();

    // parameters and conv windows: half 0 convolves q and k of channel ch, half 1 v
    const float A_h = expf(a.A_log[h]);
    const float dt_h = a.dt_bias[h];
    const float nw = a.norm_w[ch];
    const int c_a = half == 0 ? chq + ch : chv + ch;  // q (half 0) or v (half 1)
    const int c_b = chk + ch;                         // k (half 0 only)
    const float4 cwa = reinterpret_cast<const float4 *>(a.conv_w)[c_a];
    const float4 cwb = reinterpret_cast<const float4 *>(a.conv_w)[c_b];
    float wa[KM1], wb[KM1];
#pragma unroll
    for (int r = 0; r < KM1; ++r) {
        const float *row = a.conv_in + (static_cast<size_t>(b) * KM1 + r) * C;
        wa[r] = row[c_a];
        wb[r] = row[c_b];
    }
    if (clustered) cluster_arrive_relaxed();  // this CTA has read the shared q/k conv rows

    // state: S[i][j] -> TMEM S^T (lane j = ch, column i) and its split operand copy;
    // half 0 takes rows i < 64, half 1 the rest
    {
        const float *Sg = a.state_in + head * PD * PD;
        for (int i0 = 64 * half; i0 < 64 * half + 64; i0 += 16) {
            float v[16];
#pragma unroll
            for (int ii = 0; ii < 16; ++ii) v[ii] = Sg[(i0 + ii) * PD + ch];
            tc::tmem_st16(tc::taddr(tm, lb, TM_ST + i0), v);
            put_row8(st_hi, st_lo, tc::op_offset(ch, i0, PD), v);
            put_row8(st_hi, st_lo, tc::op_offset(ch, i0 + 8, PD), v + 8);
        }
    }

    // q, k, v rows of the chunk at c0: three [CH x PD] boxes of the 2-D view [B*T, C]
    auto issue_raw = [&](int c0) {
        if (lane == 0) {
            fence_proxy_async_smem();
            mbar_expect_tx(&ps.raw_full, 3 * CH * PD * 2);
            const int row = b * Ts + c0;
            tma_load_2d(raw, &tm_qkv, chq, row, &ps.raw_full);
            tma_load_2d(raw + CH * PD * 2, &tm_qkv, chk, row, &ps.raw_full);
            tma_load_2d(raw + 2 * CH * PD * 2, &tm_qkv, chv, row, &ps.raw_full);
        }
    };
    // output-gate rows of the chunk at c0: one [CH x 1 x PD] box of the 3-D view [B*T, H, PD]
    auto issue_z = [&](int c0) {
        if (lane == 0) {
            fence_proxy_async_smem();
            mbar_expect_tx(&ps.z_full, CH * PD * 2);
            tma_load_3d(zs, &tm_z, 0, h, b * Ts + c0, &ps.z_full);
        }
    };
    if (warp == 0) {
        issue_raw(0);
        issue_z(0);
    }
    // gate logits of the next chunk, one token per lane of warp 0
    float f_nx = 0.f, b_nx = 0.f;
    if (tid < CH && tid < T) {
        const size_t e = (static_cast<size_t>(b) * Ts + tid) * H + h;
        f_nx = ld_in(a.f, e, 1);
        b_nx = ld_in(a.beta, e, 1);
    }

    bool ok = true;
    uint32_t raw_ph = 0, z_ph = 0, mma_ph = 0;
    auto mma_wait = [&]() {
        if (ok) ok = mbar_wait_bounded(&ps.mma_bar, mma_ph);
        mma_ph ^= 1u;
        tc::fence_after_sync();
    };
    const int t_lo = 16 * half;  // this half's 16 tokens / columns in token-wide phases

#pragma unroll 1
    for (int c0 = 0; c0 < T; c0 += CH) {
        const int n = min(CH, T - c0);

        // P0: log-decay g, beta; G = inclusive prefix sum of g inside the chunk (warp 0)
        if (warp == 0) {
            float g = 0.f, bt = 0.f;
            if (lane < n) {
                g = -A_h * softplus_f(f_nx + dt_h);
                bt = sigmoid_f(b_nx);
            }
            if (c0 + CH + lane < T) {  // next chunk's logits, in flight during this one
                const size_t e = (static_cast<size_t>(b) * Ts + c0 + CH + lane) * H + h;
                f_nx = ld_in(a.f, e, 1);
                b_nx = ld_in(a.beta, e, 1);
            }
            float Gt = g;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, Gt, off);
                if (lane >= off) Gt += y;
            }
            ps.G[lane] = Gt;
            ps.eG[lane] = expf(Gt);
            ps.beta[lane] = bt;
        }
        if (ok) ok = mbar_wait_bounded(&ps.raw_full, raw_ph);
        raw_ph ^= 1u;
        __syncthreads();

        // P1: conv + SiLU along the chunk; half 0: split [k; q] rows, half 1: split (beta v)^T.
        // The chunk's raw values of this thread's channels are read first so the
        // conv chains of different tokens overlap.
        if (half == 0) {
            float xq[CH], xk[CH];
#pragma unroll
            for (int t = 0; t < CH; ++t) {
                xq[t] = get_bf16(raw, (0 * CH + t) * PD * 2 + ch * 2);
                xk[t] = get_bf16(raw, (1 * CH + t) * PD * 2 + ch * 2);
            }
#pragma unroll
            for (int t = 0; t < CH; ++t) {
                float q = 0.f, k = 0.f;
                if (t < n) {
                    q = conv4_silu_fast(cwa, wa, xq[t]);
                    k = conv4_silu_fast(cwb, wb, xk[t]);
                    wa[0] = wa[1]; wa[1] = wa[2]; wa[2] = xq[t];
                    wb[0] = wb[1]; wb[1] = wb[2]; wb[2] = xk[t];
                }
                put_split(r1, r1 + NR * PD * 2, tc::op_offset(t, ch, PD), k);
                put_split(r1, r1 + NR * PD * 2, tc::op_offset(CH + t, ch, PD), q);
            }
        } else {
            float xv[CH];
#pragma unroll
            for (int t = 0; t < CH; ++t) xv[t] = get_bf16(raw, (2 * CH + t) * PD * 2 + ch * 2);
            float bv[CH];
#pragma unroll
            for (int t = 0; t < CH; ++t) {
                float v = 0.f;
                if (t < n) {
                    v = conv4_silu_fast(cwa, wa, xv[t]);
                    wa[0] = wa[1]; wa[1] = wa[2]; wa[2] = xv[t];
                }
                bv[t] = ps.beta[t] * v;
            }
#pragma unroll
            for (int t0 = 0; t0 < CH; t0 += 8)
                put_row8(r2 + OP_VB, r2 + OP_VB + PD * CH * 2, tc::op_offset(ch, t0, CH), bv + t0);
        }
        publish_smem();
        if (warp == 0 && c0 + CH < T) issue_raw(c0 + CH);  // the raw stage is consumed

        // P2: Gram of the 128-row operand [k; q]_hi over [k; q]_lo with itself
        if (tid == 0) {
            tc::fence_after_sync();
            const uint32_t a1 = tc::smem_u32(r1);
            mma_chain(tm + TM_GRAM, a1, a1, PD, tc::idesc_f16(128, 2 * NR, false), false);
            tc::mma_commit(&ps.mma_bar);
        }
        mma_wait();

        // P3: exact Gram of [k; q]: hi.hi + hi.lo (rows < NR) + lo.hi (rows >= NR, via smem)
        if (quad >= 2) {
            for (int s0 = 32 * half; s0 < 32 * half + 32; s0 += 16) {
                float v[16];
                tc::tmem_ld16(tc::taddr(tm, lb, TM_GRAM + s0), v);
#pragma unroll
                for (int i = 0; i < 16; ++i) Gf[(ch - NR) * GS + s0 + i] = v[i];
            }
        }
        __syncthreads();
        if (quad < 2) {
            for (int s0 = 32 * half; s0 < 32 * half + 32; s0 += 16) {
                float hh[16], hl[16];
                tc::tmem_ld16(tc::taddr(tm, lb, TM_GRAM + s0), hh);
                tc::tmem_ld16(tc::taddr(tm, lb, TM_GRAM + NR + s0), hl);
#pragma unroll
                for (int i = 0; i < 16; ++i) Gf[ch * GS + s0 + i] += hh[i] + hl[i];
            }
        }
        __syncthreads();
        if (tid < CH) {
            ps.rk[tid] = tid < n ? 1.0f / sqrtf(Gf[tid * GS + tid] + a.eps_l2) : 0.f;
            ps.rq[tid] = tid < n ? a.q_scale / sqrtf(Gf[(CH + tid) * GS + CH + tid] + a.eps_l2) : 0.f;
        }
        __syncthreads();
        for (int e = tid; e < CH * CH; e += PT) {  // A = beta_t rk_t rk_s (k.k) e^{G_t - G_s}, s < t
            const int t = e / CH, s = e % CH;
            Af[e] = (s < t && t < n) ? ps.beta[t] * ps.rk[t] * ps.rk[s] * Gf[t * GS + s] * expf(ps.G[t] - ps.G[s]) : 0.f;
            Tf[e] = 0.f;
        }
        __syncthreads();

        // P4: T = (I + A)^-1: two 16 x 16 diagonal blocks by forward substitution, then T_10
        if (warp < 2 && lane < 16) {
            const int j = 16 * warp + lane;
            float x[16];
#pragma unroll
            for (int ii = 0; ii < 16; ++ii) {
                float acc = 0.f;
#pragma unroll
                for (int ss = 0; ss < ii; ++ss)
                    if (ss >= lane) acc = fmaf(Af[(16 * warp + ii) * CH + 16 * warp + ss], x[ss], acc);
                x[ii] = ii < lane ? 0.f : (ii == lane ? 1.f : -acc);
            }
#pragma unroll
            for (int ii = 0; ii < 16; ++ii) Tf[(16 * warp + ii) * CH + j] = x[ii];
        }
        __syncthreads();
        {  // R = A_10 T_00, one element per thread
            const int r = tid >> 4, cc = tid & 15;
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m) acc = fmaf(Af[(16 + r) * CH + m], Tf[m * CH + cc], acc);
            ps.Rt[r][cc] = acc;
        }
        __syncthreads();
        {  // T_10 = -T_11 R
            const int r = tid >> 4, cc = tid & 15;
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m) acc = fmaf(Tf[(16 + r) * CH + 16 + m], ps.Rt[m][cc], acc);
            Tf[(16 + r) * CH + cc] = -acc;
        }
        __syncthreads();
        for (int e = tid; e < CH * CH; e += PT) put_h(r4, tc::op_offset(e / CH, e % CH, CH), Tf[e]);

        // P5: operands from the split k, q rows: (beta e^G k)^T, split e^G q, split (k e^{G_last - G})^T
        const float Glast = ps.G[CH - 1];
        {
            float kbg[16], kt[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int t = t_lo + i;
                const uint32_t ok_ = tc::op_offset(t, ch, PD), oq = tc::op_offset(CH + t, ch, PD);
                const float kf = get_h(r1, ok_) + get_h(r1 + NR * PD * 2, ok_);
                const float qf = get_h(r1, oq) + get_h(r1 + NR * PD * 2, oq);
                kbg[i] = ps.beta[t] * ps.eG[t] * ps.rk[t] * kf;
                kt[i] = __expf(Glast - ps.G[t]) * ps.rk[t] * kf;
                put_split(r3 + OP_QG, r3 + OP_QG + CH * PD * 2, tc::op_offset(t, ch, PD), ps.eG[t] * ps.rq[t] * qf);
            }
            put_row8(r2 + OP_KBG, nullptr, tc::op_offset(ch, t_lo, CH), kbg);
            put_row8(r2 + OP_KBG, nullptr, tc::op_offset(ch, t_lo + 8, CH), kbg + 8);
            put_row8(r3 + OP_KT, r3 + OP_KT + PD * CH * 2, tc::op_offset(ch, t_lo, CH), kt);
            put_row8(r3 + OP_KT, r3 + OP_KT + PD * CH * 2, tc::op_offset(ch, t_lo + 8, CH), kt + 8);
        }
        publish_smem();

        // P6: W^T = (beta e^G k)^T T^T,  U^T = (beta v)^T T^T  (beta v split)
        if (tid == 0) {
            tc::fence_after_sync();
            const uint32_t id = tc::idesc_f16(128, CH, false);
            const uint32_t tb = tc::smem_u32(r4);
            mma_chain(tm + TM_WT, tc::smem_u32(r2 + OP_KBG), tb, CH, id, false);
            mma_chain(tm + TM_UT, tc::smem_u32(r2 + OP_VB), tb, CH, id, false);
            mma_chain(tm + TM_UT, tc::smem_u32(r2 + OP_VB + PD * CH * 2), tb, CH, id, true);
            tc::mma_commit(&ps.mma_bar);
        }
        mma_wait();

        // P7: split M = rq_t rk_s (q.k) e^{G_t - G_s} (s <= t); W operand [t][i] from W^T
        for (int e = tid; e < CH * CH; e += PT) {
            const int t = e / CH, s = e % CH;
            const float m = (s <= t && t < n) ? ps.rq[t] * ps.rk[s] * Gf[(CH + t) * GS + s] * expf(ps.G[t] - ps.G[s]) : 0.f;
            put_split(r2 + OP_M, r2 + OP_M + CH * CH * 2, tc::op_offset(t, s, CH), m);
        }
        {
            float w[16];
            tc::tmem_ld16(tc::taddr(tm, lb, TM_WT + t_lo), w);
#pragma unroll
            for (int i = 0; i < 16; ++i) put_h(r1, tc::op_offset(t_lo + i, ch, PD), w[i]);
        }
        publish_smem();

        // P8: V_new^T = U^T - S^T W^T  (S split)
        if (tid == 0) {
            tc::fence_after_sync();
            const uint32_t id = tc::idesc_f16(128, CH, true);
            const uint32_t bw = tc::smem_u32(r1);
            mma_chain(tm + TM_UT, tc::smem_u32(st_hi), bw, PD, id, true);
            mma_chain(tm + TM_UT, tc::smem_u32(st_lo), bw, PD, id, true);
            tc::mma_commit(&ps.mma_bar);
        }
        mma_wait();

        // P9: split V_new^T operand; S^T <- e^{G_last} S^T in TMEM
        {
            float v[16];
            tc::tmem_ld16(tc::taddr(tm, lb, TM_UT + t_lo), v);
            put_row8(r2 + OP_VN, r2 + OP_VN + PD * CH * 2, tc::op_offset(ch, t_lo, CH), v);
            put_row8(r2 + OP_VN, r2 + OP_VN + PD * CH * 2, tc::op_offset(ch, t_lo + 8, CH), v + 8);
        }
        {
            const float gam = expf(Glast);
            for (int i0 = 64 * half; i0 < 64 * half + 64; i0 += 16) {
                float sv[16];
                tc::tmem_ld16(tc::taddr(tm, lb, TM_ST + i0), sv);
#pragma unroll
                for (int i = 0; i < 16; ++i) sv[i] *= gam;
                tc::tmem_st16(tc::taddr(tm, lb, TM_ST + i0), sv);
            }
        }
        publish_smem();

        // P10: O^T = S^T (e^G q)^T + V_new^T M^T;  S^T += V_new^T (k e^{G_last - G})
        if (tid == 0) {
            tc::fence_after_sync();
            const uint32_t id32 = tc::idesc_f16(128, CH, false), id128 = tc::idesc_f16(128, PD, false);
            const uint32_t vh = tc::smem_u32(r2 + OP_VN), vl = tc::smem_u32(r2 + OP_VN + PD * CH * 2);
            mma_split(tm + TM_OT, tc::smem_u32(st_hi), tc::smem_u32(st_lo), tc::smem_u32(r3 + OP_QG),
                      tc::smem_u32(r3 + OP_QG + CH * PD * 2), PD, id32, false);
            mma_split(tm + TM_OT, vh, vl, tc::smem_u32(r2 + OP_M), tc::smem_u32(r2 + OP_M + CH * CH * 2),
                      CH, id32, true);
            mma_split(tm + TM_ST, vh, vl, tc::smem_u32(r3 + OP_KT), tc::smem_u32(r3 + OP_KT + PD * CH * 2),
                      CH, id128, true);
            tc::mma_commit(&ps.mma_bar);
        }
        mma_wait();

        // P11: gated RMSNorm over the head dimension per token; this thread holds
        // o of channel ch for tokens t_lo .. t_lo + 15
        float o[16];
        tc::tmem_ld16(tc::taddr(tm, lb, TM_OT + t_lo), o);
        float *sq = reinterpret_cast<float *>(r1);  // [CH][SQS], token-major
#pragma unroll
        for (int i = 0; i < 16; ++i) sq[(t_lo + i) * SQS + ch] = o[i] * o[i];
        __syncthreads();
        {
            const int t = tid >> 3, part = tid & 7;
            float s_ = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) s_ += sq[t * SQS + 16 * part + j];
            s_ += __shfl_xor_sync(0xffffffffu, s_, 1);
            s_ += __shfl_xor_sync(0xffffffffu, s_, 2);
            s_ += __shfl_xor_sync(0xffffffffu, s_, 4);
            if (part == 0) ps.rinv[t] = 1.0f / sqrtf(s_ / PD + a.eps_norm);
        }
        if (ok) ok = mbar_wait_bounded(&ps.z_full, z_ph);
        z_ph ^= 1u;
        __syncthreads();  // the o^2 sums are read: the scratch takes y
        // y, token-major in shared memory, then 128-bit stores of 4 channels of a token
        float *ys = reinterpret_cast<float *>(r1);  // [CH][YS]
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int t = t_lo + i;
            const float zz = get_bf16(zs, t * PD * 2 + ch * 2);
            const float gz = a.sig_gate ? __fdividef(1.0f, 1.0f + __expf(-zz)) : silu_fast(zz);
            ys[t * YS + ch] = o[i] * ps.rinv[t] * nw * gz;
        }
        __syncthreads();
#pragma unroll
        for (int k4 = 0; k4 < CH * PD / 4 / PT; ++k4) {
            const int e = tid + PT * k4, t = e / (PD / 4), c4 = 4 * (e % (PD / 4));
            if (t < n) {
                const float4 y4 = *reinterpret_cast<const float4 *>(ys + t * YS + c4);
                const size_t idx = ((static_cast<size_t>(b) * Ts + c0 + t) * H + h) * PD + c4;
                store_out4(a.out, idx, a.out_bf16, y4.x, y4.y, y4.z, y4.w);
            }
        }
        __syncthreads();  // the z stage and the scratch are consumed
        if (warp == 0 && c0 + CH < T) issue_z(c0 + CH);

        // P12: S^T -> split operand for the next chunk
        for (int i0 = 64 * half; i0 < 64 * half + 64; i0 += 16) {
            float sv[16];
            tc::tmem_ld16(tc::taddr(tm, lb, TM_ST + i0), sv);
            put_row8(st_hi, st_lo, tc::op_offset(ch, i0, PD), sv);
            put_row8(st_hi, st_lo, tc::op_offset(ch, i0 + 8, PD), sv + 8);
        }
        publish_smem();
    }

    // final state S[i][j] from S^T (lane j), and the conv window
    {
        float *So = a.state_out + head * PD * PD;
        for (int i0 = 64 * half; i0 < 64 * half + 64; i0 += 16) {
            float sv[16];
            tc::tmem_ld16(tc::taddr(tm, lb, TM_ST + i0), sv);
#pragma unroll
            for (int i = 0; i < 16; ++i) So[(i0 + i) * PD + ch] = sv[i];
        }
    }
    if (clustered) cluster_wait_acquire();  // every CTA of the group has read the q/k rows
#pragma unroll
    for (int r = 0; r < KM1; ++r) {
        float *row = a.conv_out + (static_cast<size_t>(b) * KM1 + r) * C;
        if (half == 0) {
            if (qk_owner) {
                row[c_a] = wa[r];
                row[c_b] = wb[r];
            }
        } else {
            row[c_a] = wa[r];
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, 512);
    if (!ok && lane == 0) atomicOr(&g_prefill_error, 1u);
}

// Shapes the single tensor-core kernel takes (its pointer rules aside): the caller
// asks for its 32-token chunks with chunk == 32; other chunk lengths take the
// faster two-kernel form (gdn_kda_prefill.cu).
bool chunked_shape(const gdn_shape_t &s)
{
    const int group = s.H_v / s.H_qk;
    const size_t C = 2 * static_cast<size_t>(s.H_qk) * s.d_k + static_cast<size_t>(s.H_v) * s.d_v;
    return s.gate_mode == GDN_GATE_PER_HEAD && s.d_k == PD && s.d_v == PD &&
           s.in_dtype == GDN_BF16 && s.chunk == CH && group <= 8 &&
           (C * 2) % 16 == 0 && static_cast<long long>(s.B) * s.T < (1LL << 31);
}

bool chunked_eligible(const gdn_shape_t &s, const StepArgs &a)
{
    return chunked_shape(s) && (reinterpret_cast<uintptr_t>(a.qkv) & 15u) == 0 &&
           (reinterpret_cast<uintptr_t>(a.z) & 15u) == 0;
}

// Shapes that run the two-kernel chunked form over a workspace.
bool two_stage_shape(const gdn_shape_t &s)
{
    return !chunked_shape(s) && !c64_shape(s) && kda_chunk_shape(s);
}

cudaError_t launch_chunked(const StepArgs &a, cudaStream_t stream)
{
    static bool attr_set[64];  // per device; benign race: every writer sets the same value
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(chunk_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    CUtensorMap tq, tz;
    const uint64_t rows = static_cast<uint64_t>(a.B) * a.Ts;
    {   // qkv as [B*T rows][C channels] bf16, boxes of CH rows x PD channels
        const uint64_t dim[2] = {static_cast<uint64_t>(a.C), rows};
        const uint64_t stride[1] = {static_cast<uint64_t>(a.C) * 2};
        const uint32_t box[2] = {PD, CH};
        if (!encode_tiled(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.qkv, dim, stride, box))
            return cudaErrorInvalidValue;
    }
    {   // z as [B*T][H_v][PD] bf16, boxes of CH tokens x 1 head x PD channels
        const uint64_t dim[3] = {PD, static_cast<uint64_t>(a.H_v), rows};
        const uint64_t stride[2] = {PD * 2, static_cast<uint64_t>(a.H_v) * PD * 2};
        const uint32_t box[3] = {PD, 1, CH};
        if (!encode_tiled(&tz, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.z, dim, stride, box))
            return cudaErrorInvalidValue;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.H_v, a.B, 1);
    cfg.blockDim = dim3(PT, 1, 1);
    cfg.dynamicSmemBytes = SM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    int n = 0;
    if (a.group > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = a.group;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, chunk_prefill_kernel, a, tq, tz);
}

}  // namespace

size_t prefill_workspace_bytes(const gdn_shape_t &s)
{
    return two_stage_shape(s) ? kda_chunk_workspace_bytes(s) : 0;
}

const char *prefill_variant(const gdn_shape_t &s, int num_sms)
{
    if (chunked_shape(s)) return "chunked<128,32>";
    if (c64_shape(s)) return "chunked<128,64>";
    if (two_stage_shape(s)) return "kda_chunked<16>";
    StepPlan plan;
    const int sms = num_sms > 0 ? num_sms : 148;
    const bool planned = s.T <= 4 ? plan_step(s.d_k, s.B, s.H_v, s.H_v / s.H_qk, sms, &plan)
                                  : plan_slab_one_wave(s.d_k, s.B, s.H_v, s.H_v / s.H_qk, sms, &plan);
    return planned ? plan.name : nullptr;
}

gdn_status_t run_prefill(const gdn_shape_t &s, const StepArgs &a, void *workspace, int num_sms,
                         cudaStream_t stream)
{
    if (c64_shape(s) && c64_pointers_ok(a)) {
        cudaError_t e = launch_c64(a, stream);
        return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
    }
    if (chunked_eligible(s, a)) {
        cudaError_t e = launch_chunked(a, stream);
        return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
    }
    if (two_stage_shape(s) && kda_chunk_pointers_ok(a)) {
        cudaError_t e = launch_kda_chunked(a, workspace, stream);
        return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
    }
    // the recurrent kernel over all T tokens: short runs take the step plan, long ones the
    // column-slab plan that is resident in one wave
    StepPlan plan;
    const bool planned = s.T <= 4 ? plan_step(s.d_k, s.B, s.H_v, s.H_v / s.H_qk, num_sms, &plan)
                                  : plan_slab_one_wave(s.d_k, s.B, s.H_v, s.H_v / s.H_qk, num_sms, &plan);
    if (!planned) return GDN_ERR_UNSUPPORTED;
    cudaError_t e = launch_step(plan, a, (s.flags & GDN_FLAG_PDL) != 0, num_sms, stream);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status_t run_prefill_snapshots(const gdn_shape_t &s, const StepArgs &a, void *workspace,
                                   int num_sms, cudaStream_t stream)
{
    const int n = s.T < 4 ? s.T : 4, Tm = s.T - n;
    if (Tm > 0) {  // the head of each sequence: rows 0 .. Tm - 1 of the [B, T, ...] tensors
        gdn_shape_t sm = s;
        sm.T = Tm;
        StepArgs am = a;
        am.T = Tm;
        am.state_hist = nullptr;
        am.conv_hist = nullptr;
        const gdn_status_t rc = run_prefill(sm, am, workspace, num_sms, stream);
        if (rc != GDN_OK) return rc;
    }
    // the tail: rows Tm .. T - 1, from the state and window the head left in place
    const size_t es = a.in_bf16 ? 2 : 4, os = a.out_bf16 ? 2 : 4, d = s.d_k;
    const size_t fw = a.kda ? d : 1;
    StepArgs at = a;
    at.T = n;
    at.Ts = s.T;
    at.qkv = static_cast<const char *>(a.qkv) + static_cast<size_t>(Tm) * a.C * es;
    at.f = static_cast<const char *>(a.f) + static_cast<size_t>(Tm) * a.H_v * fw * es;
    at.beta = static_cast<const char *>(a.beta) + static_cast<size_t>(Tm) * a.H_v * es;
    at.z = static_cast<const char *>(a.z) + static_cast<size_t>(Tm) * a.H_v * d * es;
    at.out = static_cast<char *>(a.out) + static_cast<size_t>(Tm) * a.H_v * d * os;
    at.state_in = a.state_out;
    at.conv_in = a.conv_out;
    at.accepted = nullptr;
    StepPlan plan;
    if (!plan_slab(s.d_k, s.B, s.H_v, s.H_v / s.H_qk, num_sms, &plan)) return GDN_ERR_UNSUPPORTED;
    // plain stream order: the head (when there is one) writes the state the tail reads first
    const bool pdl = Tm == 0 && (s.flags & GDN_FLAG_PDL) != 0;
    const cudaError_t e = launch_slab(plan, at, pdl, stream);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

unsigned int take_prefill_error()
{
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_prefill_error, sizeof(v)) != cudaSuccess) return ~0u;
    if (v && cudaMemcpyToSymbol(g_prefill_error, &zero, sizeof(zero)) != cudaSuccess) return ~0u;
    return v;
}

}  // namespace gdn
