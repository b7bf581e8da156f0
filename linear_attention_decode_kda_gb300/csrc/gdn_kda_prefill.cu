// Chunked prefill for the per-channel decay (KDA), and for per-head decay shapes
// the single-kernel tensor-core prefill does not take: two kernels over a
// device workspace.
//
// The form is the chunked WY/UT recurrence with one log-decay per key channel,
// split the way "llama.cpp PR #84" splits its chunked KDA prefill (an intra-chunk
// stage that needs no state, then a state stage over the chunks).  Inside a chunk
// of KC = 16 tokens with start state S0, G[t][i] is channel i's log-decay summed
// from the chunk's first token through t, so every exponent below is <= 0:
//   L[t][s] = beta_t sum_i k[t][i] k[s][i] e^{G[t][i] - G[s][i]}      (s < t)
//   A[t][s] = sum_i q[t][i] k[s][i] e^{G[t][i] - G[s][i]}             (s <= t)
//   W = (I + L)^-1 (beta e^G * K),  U = (I + L)^-1 (beta V)
//   V_new = U - W S0,   O = (e^G * Q) S0 + A V_new
//   S = Diag(e^{G_last}) S0 + (e^{G_last - G} * K)^T V_new
// (G_last = G of the chunk's last token; q, k are the L2-normalised rows, q
// scaled.)  The per-token form it restates is the step of "Thirty tiny kernels
// per layer"; T of these steps and this form agree up to rounding.
//
// kda_intra_kernel: one CTA per (sequence, head, chunk), all chunks at once,
// on the CUDA cores (the pair sums need an exponential per element).  It runs
// the conv, the norms, the gates, L and A and the forward substitution, and
// writes one block per chunk: the tensor-core operands W, e^G * Q,
// (e^{G_last - G} * K)^T and A as fp16 hi/lo pairs, U and e^{G_last} in fp32.
// kda_state_kernel: one CTA per (sequence, head) carries S through the chunks
// on tcgen05.  S^T (lane = state column) is the fp32 accumulator in TMEM, with
// a split-fp16 copy in shared memory as the A operand; per chunk
//   P^T = S^T W^T                      -> V_new = U - P on the CUDA cores
//   O^T = S^T (e^G Q)^T + V_new^T A^T,  S^T = e^{G_last} S^T + V_new^T (e^{G_last-G} K)
// then the gated RMSNorm and the output store.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"
#include "gdn_device.cuh"
#include "gdn_internal.h"
#include "gdn_prefill.h"
#include "gdn_tc.cuh"
#include "gdn_tmap.h"

namespace gdn {
namespace {

using namespace dev;

constexpr int KD = 128;  // d_k = d_v
constexpr int KC = 16;   // tokens per chunk
// Workspace block of one (sequence, head, chunk), in bytes.  Tensor-core
// operands are fp16 hi/lo pairs in the canonical K-major layout (tc::op_offset).
constexpr int BW_WQ = 0;     // [W; e^G Q] [32 rows][128 i] (W rows 0-15): hi (8 KiB), then lo
constexpr int BW_K = 16384;  // (e^{G_last - G} K)^T [128 i][16 t]: hi, lo
constexpr int BW_M = 24576;  // A [16 t][16 s]: hi (512 B), then lo
constexpr int BW_U = 25600;  // U [16 t][128 j], fp32
constexpr int BW_G = 33792;  // e^{G_last} [128], fp32
constexpr uint32_t BLOCK_BYTES = 34304;
static_assert(BW_G + KD * 4 == BLOCK_BYTES, "block layout");
static_assert(BLOCK_BYTES % 16 == 0, "bulk copies move multiples of 16 bytes");

__device__ unsigned int g_kda_error;

// Intra kernel staging rows: 136 floats, 4 spare after channel 63, so the two
// channel halves of a row sit in different banks.
constexpr int SP = 136;
// fp32 rows of [W; e^G Q] before their split into the canonical layout: a stride of
// 132 floats (4 banks on a row) lets 8 rows' 16-byte pieces be read without conflict.
constexpr int FS = 132;
// dynamic shared memory of the intra kernel: the staging rows, then the W/Q rows
constexpr int INTRA_STG = 4 * KC * SP * 4;
constexpr int INTRA_SMEM = INTRA_STG + 2 * KC * FS * 4;
__device__ __forceinline__ int hp(int i) { return i + ((i >> 6) << 2); }

// SiLU and sigmoid on the fast exponential and division: within a few units in
// the last place of fp32, far inside the prefill's tolerance.
__device__ __forceinline__ float fast_sigmoid(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }
__device__ __forceinline__ float fast_silu(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

// 2^x and log2(x) on the hardware approximations (relative error about 2^-22).
// The intra kernel keeps the cumulative log-decays in log2 units, so every decay
// factor it forms is one ex2 of a difference <= 0.
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float2 lo2(const float4 v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 hi2(const float4 v) { return make_float2(v.z, v.w); }

// After the call lane l holds the warp-wide sum of v[l].
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane)
{
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) {
        const bool up = (lane & w) != 0;
#pragma unroll
        for (int j = 0; j < w; ++j) {
            const float send = up ? v[j] : v[j + w];
            const float keep = up ? v[j + w] : v[j];
            v[j] = keep + __shfl_xor_sync(0xffffffffu, send, w);
        }
    }
    return v[0];
}

// bf16 rows t0 - 3 .. t0 + 15 of one head's q, k and v channels: three TMA
// boxes of 19 rows x 128 channels, then the chunk's 16 gate rows (per-channel
// gates), laid over the staging rows until the conv has read them.
constexpr int RAW_ROWS = KC + 3;
constexpr int RAW_SEG = RAW_ROWS * KD * 2;  // bytes of one box (a multiple of 128)
static_assert(RAW_SEG % 128 == 0, "TMA destinations 128-byte aligned");

template <bool BF16, bool PER_CHANNEL>
__global__ void __launch_bounds__(256, 4)
kda_intra_kernel(StepArgs a, unsigned char *ws, const __grid_constant__ CUtensorMap tq,
                 const __grid_constant__ CUtensorMap tf)
{
    // staging rows of q, k, v and G; they take the block image at the end
    extern __shared__ __align__(1024) unsigned char ism[];
    float(*stg)[KC][SP] = reinterpret_cast<float(*)[KC][SP]>(ism);
    float(*fwq)[FS] = reinterpret_cast<float(*)[FS]>(ism + INTRA_STG);
    __shared__ uint64_t raw_bar;
    float(*qs)[SP] = stg[0];
    float(*ks)[SP] = stg[1];
    float(*vs)[SP] = stg[2];
    float(*gs)[SP] = stg[3];
    __shared__ __align__(16) float Ls[KC][KC];
    __shared__ __align__(16) float As[KC][KC];
    __shared__ float bs[KC];
    __shared__ float red[4][32];
    __shared__ float rqk[2][KC];  // per token: q_scale / |q|, 1 / |k|

    const int n = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int i = tid & (KD - 1);
    const int t0 = n * KC;
    const int nt = min(KC, a.T - t0);
    const int hq = h / a.group;
    const size_t C = static_cast<size_t>(a.C);
    const size_t row0 = static_cast<size_t>(b) * a.Ts + t0;
    auto ld = [&](const void *p, size_t idx) {
        return BF16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[idx])
                    : reinterpret_cast<const float *>(p)[idx];
    };

    // channel c's rows t0 - 3 .. t0 + 15: the three before t0 come from the
    // sequence, or from the kept window before its start; rows past the
    // sequence repeat its last row (their outputs are zeroed)
    auto load_rows = [&](int c, float(&x)[KC + 3]) {
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const int tau = t0 - 3 + j;
            x[j] = tau >= 0 ? ld(a.qkv, (static_cast<size_t>(b) * a.Ts + tau) * C + c)
                            : a.conv_in[(static_cast<size_t>(b) * 3 + (3 + tau)) * C + c];
        }
        const size_t base = static_cast<size_t>(b) * a.Ts;
#pragma unroll
        for (int t = 0; t < KC; ++t) x[3 + t] = ld(a.qkv, (base + min(t0 + t, a.T - 1)) * C + c);
    };
    // 4-tap causal conv + SiLU of those rows
    auto conv_rows = [&](int c, const float(&x)[KC + 3], float(&y)[KC]) {
        const float4 w = reinterpret_cast<const float4 *>(a.conv_w)[c];
#pragma unroll
        for (int t = 0; t < KC; ++t) {
            float acc = w.x * x[t];
            acc = fmaf(w.y, x[t + 1], acc);
            acc = fmaf(w.z, x[t + 2], acc);
            acc = fmaf(w.w, x[t + 3], acc);
            y[t] = t < nt ? fast_silu(acc) : 0.f;
        }
    };

    // bf16 rows by TMA; fp32 rows (and the per-head gate) by plain loads
    const unsigned char *raw = reinterpret_cast<const unsigned char *>(&stg[0][0][0]);
    const int chq = hq * KD, chk = a.H_qk * KD + hq * KD, chv = 2 * a.H_qk * KD + h * KD;
    if (BF16) {
        if (tid == 0) {
            mbar_init(&raw_bar, 1);
            fence_mbar_init();
        }
        __syncthreads();
        if (tid == 0) {
            unsigned char *dst = reinterpret_cast<unsigned char *>(&stg[0][0][0]);
            const int row = b * a.Ts + t0 - 3;  // rows before the batch read as zero
            mbar_expect_tx(&raw_bar, 3 * RAW_SEG + (PER_CHANNEL ? KC * KD * 2 : 0));
            tma_load_2d(dst, &tq, chq, row, &raw_bar);
            tma_load_2d(dst + RAW_SEG, &tq, chk, row, &raw_bar);
            tma_load_2d(dst + 2 * RAW_SEG, &tq, chv, row, &raw_bar);
            if (PER_CHANNEL) tma_load_3d(dst + 3 * RAW_SEG, &tf, 0, h, b * a.Ts + t0, &raw_bar);
        }
    }
    // channel i of box sg: rows t0 - 3 .. t0 + 15, the first three from the kept
    // window at the sequence's start
    auto box_rows = [&](int sg, int c, float(&x)[KC + 3]) {
        const __nv_bfloat16 *r = reinterpret_cast<const __nv_bfloat16 *>(raw + sg * RAW_SEG) + i;
#pragma unroll
        for (int j = 0; j < KC + 3; ++j) x[j] = __bfloat162float(r[j * KD]);
        if (t0 == 0)
#pragma unroll
            for (int j = 0; j < 3; ++j) x[j] = a.conv_in[(static_cast<size_t>(b) * 3 + j) * C + c];
    };

    // ---- 1. conv, squares for the L2 norms, gates; padded tokens are zero
    if (tid < KC) bs[tid] = tid < nt ? fast_sigmoid(ld(a.beta, (row0 + tid) * a.H_v + h)) : 0.f;
    Ls[tid >> 4][tid & 15] = 0.f;
    As[tid >> 4][tid & 15] = 0.f;
    float fl[KC];
    if (tid >= KD && !(BF16 && PER_CHANNEL)) {
#pragma unroll
        for (int t = 0; t < KC; ++t) {
            const size_t bth = (static_cast<size_t>(b) * a.Ts + min(t0 + t, a.T - 1)) * a.H_v + h;
            fl[t] = PER_CHANNEL ? ld(a.f, bth * KD + i) : ld(a.f, bth);
        }
    }
    if (BF16 && !mbar_wait_bounded(&raw_bar, 0)) atomicOr(&g_kda_error, 1u);
    float q[KC], k[KC], v[KC];
    if (tid < KD) {
        float xq[KC + 3], xk[KC + 3];
        if (BF16) {
            box_rows(0, chq + i, xq);
            box_rows(1, chk + i, xk);
        } else {
            load_rows(chq + i, xq);
            load_rows(chk + i, xk);
        }
        conv_rows(chq + i, xq, q);
        conv_rows(chk + i, xk, k);
    } else {
        float xv[KC + 3];
        if (BF16) {
            box_rows(2, chv + i, xv);
            if (PER_CHANNEL)
#pragma unroll
                for (int t = 0; t < KC; ++t)
                    fl[t] = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(raw + 3 * RAW_SEG)[t * KD + i]);
        } else {
            load_rows(chv + i, xv);
        }
        conv_rows(chv + i, xv, v);
    }
    if (BF16) __syncthreads();  // the rows are read: the staging rows take q, k, v, G
    if (tid < KD) {
        float sq2[32];
#pragma unroll
        for (int t = 0; t < KC; ++t) {
            sq2[t] = q[t] * q[t];
            sq2[KC + t] = k[t] * k[t];
            qs[t][hp(i)] = q[t];  // raw rows; the norms scale the products below
            ks[t][hp(i)] = k[t];
        }
        red[warp][lane] = reduce_scatter32(sq2, lane);
    } else {
#pragma unroll
        for (int t = 0; t < KC; ++t) vs[t][hp(i)] = v[t];
        // log-decays of channel i summed along the chunk, in log2 units.  Softplus
        // gates: g = -exp(A_log) softplus(f + dt_bias), with softplus(x) = max(x, 0)
        // + ln(1 + e^-|x|); lower-bound gate: g = lb sigmoid(-a f)
        const float A = a.lb_gate ? a.A_log[h] : expf(a.A_log[h]);
        const float lbv = a.lb_gate ? a.dt_bias[h] * kLog2e : 0.f;
        const float dtb = a.lb_gate ? 0.f : (a.kda ? a.dt_bias[static_cast<size_t>(h) * KD + i] : a.dt_bias[h]);
        float G = 0.f;
#pragma unroll
        for (int t = 0; t < KC; ++t) {
            const float x = fl[t] + dtb;
            const float g2 = a.lb_gate ? lbv * fast_sigmoid(-A * fl[t])
                                       : -A * fmaf(fmaxf(x, 0.f), kLog2e, lg2(1.0f + ex2(-fabsf(x) * kLog2e)));
            if (t < nt) G += g2;
            gs[t][hp(i)] = G;
        }
    }
    __syncthreads();
    if (tid < 32) {  // the L2 norms: lanes 0-15 q of token lane, 16-31 k of token lane - 16
        const float sq = red[0][tid] + red[1][tid] + red[2][tid] + red[3][tid];
        rqk[tid >> 4][tid & 15] = (tid < KC ? a.q_scale : 1.0f) / sqrtf(sq + a.eps_l2);
    }
    __syncthreads();

    // ---- 2. pair sums: thread pairs split (t, s), s < t, over the two channel
    // halves; the last 16 threads take the diagonal q_t . k_t
    {
        int t = 0, s = 0;
        float kk = 0.f, qk = 0.f;
        if (tid < 240) {
            int p = tid >> 1;
            t = 1;
            while (p >= t) {
                p -= t;
                ++t;
            }
            s = p;
            const int base = 68 * (tid & 1);
            // two channels at a time on the packed fp32 pipe
            float2 kk2 = make_float2(0.f, 0.f), qk2 = kk2;
            const float2 neg1 = make_float2(-1.f, -1.f);
            if (!PER_CHANNEL) {
                // one decay per head: e^{G_t - G_s} factors out of the channel sums
#pragma unroll 4
                for (int m = 0; m < 64; m += 4) {
                    const float4 k1 = *reinterpret_cast<const float4 *>(&ks[t][base + m]);
                    const float4 k0 = *reinterpret_cast<const float4 *>(&ks[s][base + m]);
                    const float4 q1 = *reinterpret_cast<const float4 *>(&qs[t][base + m]);
                    kk2 = __ffma2_rn(lo2(k1), lo2(k0), kk2);
                    qk2 = __ffma2_rn(lo2(q1), lo2(k0), qk2);
                    kk2 = __ffma2_rn(hi2(k1), hi2(k0), kk2);
                    qk2 = __ffma2_rn(hi2(q1), hi2(k0), qk2);
                }
                const float e = ex2(gs[t][0] - gs[s][0]);
                kk2 = make_float2(kk2.x * e, kk2.y * e);
                qk2 = make_float2(qk2.x * e, qk2.y * e);
            } else
#pragma unroll 4
            for (int m = 0; m < 64; m += 4) {
                const float4 g1 = *reinterpret_cast<const float4 *>(&gs[t][base + m]);
                const float4 g0 = *reinterpret_cast<const float4 *>(&gs[s][base + m]);
                const float4 k1 = *reinterpret_cast<const float4 *>(&ks[t][base + m]);
                const float4 k0 = *reinterpret_cast<const float4 *>(&ks[s][base + m]);
                const float4 q1 = *reinterpret_cast<const float4 *>(&qs[t][base + m]);
                const float2 dl = __ffma2_rn(lo2(g0), neg1, lo2(g1)), dh = __ffma2_rn(hi2(g0), neg1, hi2(g1));
                const float2 el = make_float2(ex2(dl.x), ex2(dl.y)), eh = make_float2(ex2(dh.x), ex2(dh.y));
                kk2 = __ffma2_rn(__fmul2_rn(lo2(k1), lo2(k0)), el, kk2);
                qk2 = __ffma2_rn(__fmul2_rn(lo2(q1), lo2(k0)), el, qk2);
                kk2 = __ffma2_rn(__fmul2_rn(hi2(k1), hi2(k0)), eh, kk2);
                qk2 = __ffma2_rn(__fmul2_rn(hi2(q1), hi2(k0)), eh, qk2);
            }
            kk = kk2.x + kk2.y;
            qk = qk2.x + qk2.y;
        } else {
            t = tid - 240;
#pragma unroll 4
            for (int m = 0; m < KD; m += 4) {
                const float4 q1 = *reinterpret_cast<const float4 *>(&qs[t][hp(m)]);
                const float4 k1 = *reinterpret_cast<const float4 *>(&ks[t][hp(m)]);
                qk = fmaf(q1.x, k1.x, qk);
                qk = fmaf(q1.y, k1.y, qk);
                qk = fmaf(q1.z, k1.z, qk);
                qk = fmaf(q1.w, k1.w, qk);
            }
        }
        const float kk2 = __shfl_xor_sync(0xffffffffu, kk, 1);
        const float qk2 = __shfl_xor_sync(0xffffffffu, qk, 1);
        if (tid < 240) {
            if ((tid & 1) == 0) {
                Ls[t][s] = bs[t] * (kk + kk2) * rqk[1][t] * rqk[1][s];
                As[t][s] = (qk + qk2) * rqk[0][t] * rqk[1][s];
            }
        } else {
            As[t][t] = qk * rqk[0][t] * rqk[1][t];
        }
    }
    __syncthreads();

    // ---- 3. (I + L) X = B by forward substitution, one column a thread: W's
    // columns from beta e^G k (threads 0-127), U's from beta v (128-255); then the
    // block image in shared memory over the staging rows, copied out coalesced
    float x[KC], y[KC], gl = 0.f;
    {
        const bool wside = tid < KD;
#pragma unroll
        for (int t = 0; t < KC; ++t)
            x[t] = bs[t] * (wside ? ks[t][hp(i)] * rqk[1][t] * ex2(gs[t][hp(i)]) : vs[t][hp(i)]);
#pragma unroll
        for (int t = 1; t < KC; ++t) {
            float l[KC];
#pragma unroll
            for (int s4 = 0; s4 < KC; s4 += 4) {
                const float4 v4 = *reinterpret_cast<const float4 *>(&Ls[t][s4]);
                l[s4] = v4.x;
                l[s4 + 1] = v4.y;
                l[s4 + 2] = v4.z;
                l[s4 + 3] = v4.w;
            }
#pragma unroll
            for (int s = 0; s < t; ++s) x[t] = fmaf(-l[s], x[s], x[t]);
        }
        if (wside) {
#pragma unroll
            for (int t = 0; t < KC; ++t) y[t] = qs[t][hp(i)] * rqk[0][t] * ex2(gs[t][hp(i)]);
        } else {
            const float Gl = gs[KC - 1][hp(i)];
#pragma unroll
            for (int t = 0; t < KC; ++t) y[t] = ks[t][hp(i)] * rqk[1][t] * ex2(Gl - gs[t][hp(i)]);
            gl = ex2(Gl);
        }
    }
    const float m = As[tid >> 4][tid & 15];
    if (tid < KD)
#pragma unroll
        for (int t = 0; t < KC; ++t) {
            fwq[t][i] = x[t];
            fwq[KC + t][i] = y[t];
        }
    __syncthreads();  // the staging rows are read: they take the block image
    unsigned char *img = reinterpret_cast<unsigned char *>(&stg[0][0][0]);
    if (tid < KD) {
        // [W; e^G Q] split into fp16 hi/lo: one 8-row x 8-channel core matrix per 8
        // threads (8 rows of one channel group), 16-byte reads and writes
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int r = 8 * e + (tid & 7), c8 = 8 * (tid >> 3);
            float v8[8];
            const float4 u0 = *reinterpret_cast<const float4 *>(&fwq[r][c8]);
            const float4 u1 = *reinterpret_cast<const float4 *>(&fwq[r][c8 + 4]);
            v8[0] = u0.x; v8[1] = u0.y; v8[2] = u0.z; v8[3] = u0.w;
            v8[4] = u1.x; v8[5] = u1.y; v8[6] = u1.z; v8[7] = u1.w;
            tc::put_row8(img + BW_WQ, img + BW_WQ + 8192, tc::op_offset(r, c8, KD), v8);
        }
    } else {
        float *U = reinterpret_cast<float *>(img + BW_U);
#pragma unroll
        for (int t = 0; t < KC; ++t) U[t * KD + i] = x[t];
        tc::put_row8(img + BW_K, img + BW_K + 4096, tc::op_offset(i, 0, KC), y);
        tc::put_row8(img + BW_K, img + BW_K + 4096, tc::op_offset(i, 8, KC), y + 8);
        reinterpret_cast<float *>(img + BW_G)[i] = gl;
    }
    tc::put_split(img + BW_M, img + BW_M + 512, tc::op_offset(tid >> 4, tid & 15, KC), m);
    __syncthreads();
    uint4 *dst = reinterpret_cast<uint4 *>(
        ws + ((static_cast<size_t>(b) * a.H_v + h) * gridDim.x + n) * BLOCK_BYTES);
    const uint4 *src = reinterpret_cast<const uint4 *>(img);
    for (int e = tid; e < static_cast<int>(BLOCK_BYTES / 16); e += 256) dst[e] = src[e];
}

// ---------------------------------------------------------------- state stage

constexpr int NSTG = 3;
// A stage holds the chunk's block, then its 16 output-gate rows (z, in dtype).
constexpr int STAGE_Z = 34816;             // block bytes rounded up to 1 KiB
constexpr int STAGE = STAGE_Z + KC * KD * 4;
static_assert(STAGE_Z >= static_cast<int>(BLOCK_BYTES) && STAGE % 1024 == 0, "stage size");
// TMEM columns
constexpr int TM_S = 0;     // 128: S^T (lane j = state column j, column i = state row i)
constexpr int TM_P = 128;   // 16: P^T = (W S)^T
constexpr int TM_O = 144;   // 16: (e^G Q S)^T, then O^T
constexpr uint32_t TM_COLS = 256;
// dynamic shared memory (bytes)
constexpr int SS_ST = NSTG * STAGE;             // split S^T [128 j][128 i]: hi (32 KiB), lo
constexpr int SS_VN = SS_ST + 2 * KD * KD * 2;  // split V_new^T [128 j][16 t]: hi (4 KiB), lo
constexpr int SS_SQ = SS_VN + 2 * KD * KC * 2;  // o^2 [16 t][SQS]
constexpr int SQS = KD + 4;
constexpr int SS_BYTES = SS_SQ + KC * SQS * 4;

struct StateShared {
    float rinv[KC];
    uint64_t full[NSTG];
    uint64_t mma_bar;
    uint32_t tmem;
    int fail;  // a bounded wait gave up somewhere in the CTA
};

// Makes this thread's shared-memory writes visible to the tensor core, then syncs the CTA.
__device__ __forceinline__ void publish_smem()
{
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
}

constexpr int CT = 256;           // compute threads (8 warps)
constexpr int ST_THREADS = CT + 32;  // plus the issuing warp
constexpr int ISSUER_WARP = CT / 32;

// Named barrier of the 256 compute threads (the norm's partial sums).
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
// The CTA-wide barrier, taken by the compute warps and the issuing warp alike.
__device__ __forceinline__ void cta_sync() { asm volatile("bar.sync 0;" ::: "memory"); }

// A shared-memory descriptor moved `bytes` further (the start address sits in
// bits 0-13 in 16-byte units; every operand here lies below 256 KiB).
__device__ __forceinline__ uint64_t desc_at(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

// Warps 0-7: ch = tid % 128 is the state column j (TMEM lane j, warp w reaching
// lanes 32 (w % 4) ..); half = tid / 128 splits the row-wise work.  Warp 8 issues
// every copy and every product, with descriptors computed once, so issuing never
// sits on the compute warps' path.
__global__ void __launch_bounds__(ST_THREADS, 1)
kda_state_kernel(StepArgs a, const unsigned char *ws, int nchunk, const __grid_constant__ CUtensorMap tmz)
{
    extern __shared__ __align__(1024) unsigned char sm[];
    __shared__ __align__(16) StateShared ps;
    const int h = blockIdx.x, b = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool issuer = warp == ISSUER_WARP;
    const int ch = tid & (KD - 1), half = (tid >> 7) & 1;
    const int lb = 32 * (warp & 3);
    const size_t head = static_cast<size_t>(b) * a.H_v + h;
    const unsigned char *blocks = ws + head * nchunk * static_cast<size_t>(BLOCK_BYTES);
    unsigned char *st_hi = sm + SS_ST, *st_lo = sm + SS_ST + KD * KD * 2;
    unsigned char *vn_hi = sm + SS_VN, *vn_lo = sm + SS_VN + KD * KC * 2;
    float *sq = reinterpret_cast<float *>(sm + SS_SQ);

    if (warp == 0) tc::tmem_alloc(&ps.tmem, TM_COLS);
    if (tid == 0) {
        for (int s = 0; s < NSTG; ++s) mbar_init(&ps.full[s], 1);
        mbar_init(&ps.mma_bar, 1);
        ps.fail = 0;
        fence_mbar_init();
    }
    tc::fence_before_sync();
    cta_sync();
    tc::fence_after_sync();
    const uint32_t tm = ps.tmem;
    bool ok = true;

    if (issuer) {
        const uint32_t zbytes = KC * KD * (a.in_bf16 ? 2u : 4u);
        auto issue = [&](int n) {
            const int s = n % NSTG;
            mbar_expect_tx(&ps.full[s], BLOCK_BYTES + zbytes);
            tma_load_1d(sm + s * STAGE, blocks + static_cast<size_t>(n) * BLOCK_BYTES, BLOCK_BYTES, &ps.full[s]);
            // rows past the last token of the batch read as zero; rows of the next sequence are unused
            tma_load_3d(sm + s * STAGE + STAGE_Z, &tmz, 0, h, b * a.Ts + n * KC, &ps.full[s]);
        };
        // descriptors: S^T (A, K = 128) and stage 0's [W; e^G Q] (B, K = 128); the
        // K = 16 operands V_new^T (A), A (B) and (e^{G_last-G} K)^T (B)
        uint64_t dsh[8], dsl[8], dwh[8], dwl[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            dsh[i] = tc::op_desc(tc::smem_u32(st_hi), 16 * i, KD);
            dsl[i] = tc::op_desc(tc::smem_u32(st_lo), 16 * i, KD);
            dwh[i] = tc::op_desc(tc::smem_u32(sm + BW_WQ), 16 * i, KD);
            dwl[i] = tc::op_desc(tc::smem_u32(sm + BW_WQ + 8192), 16 * i, KD);
        }
        const uint64_t dvh = tc::op_desc(tc::smem_u32(vn_hi), 0, KC), dvl = tc::op_desc(tc::smem_u32(vn_lo), 0, KC);
        const uint64_t dmh = tc::op_desc(tc::smem_u32(sm + BW_M), 0, KC),
                       dml = tc::op_desc(tc::smem_u32(sm + BW_M + 512), 0, KC);
        const uint64_t dkh = tc::op_desc(tc::smem_u32(sm + BW_K), 0, KC),
                       dkl = tc::op_desc(tc::smem_u32(sm + BW_K + 4096), 0, KC);
        const uint32_t id16 = tc::idesc_f16(128, KC, false), id32 = tc::idesc_f16(128, 2 * KC, false),
                       id128 = tc::idesc_f16(128, KD, false);
        // 1. [P | Q']^T = S^T [W; e^G Q]^T of chunk n (one N = 32 product, split operands)
        auto issue_p = [&](int n) {
            const uint32_t so = (n % NSTG) * STAGE;
            if (ok) ok = mbar_wait_bounded(&ps.full[n % NSTG], static_cast<uint32_t>((n / NSTG) & 1));
            tc::fence_after_sync();
#pragma unroll
            for (int i = 0; i < 8; ++i) tc::mma_f16(tm + TM_P, dsh[i], desc_at(dwh[i], so), id32, i > 0);
#pragma unroll
            for (int i = 0; i < 8; ++i) tc::mma_f16(tm + TM_P, dsh[i], desc_at(dwl[i], so), id32, true);
#pragma unroll
            for (int i = 0; i < 8; ++i) tc::mma_f16(tm + TM_P, dsl[i], desc_at(dwh[i], so), id32, true);
            tc::mma_commit(&ps.mma_bar);
        };
        // 3. O^T = Q'^T + V_new^T A^T;  S^T += V_new^T (e^{G_last - G} K)
        auto issue_o = [&](int n) {
            const uint32_t so = (n % NSTG) * STAGE;
            tc::fence_after_sync();
            tc::mma_f16(tm + TM_O, dvh, desc_at(dmh, so), id16, true);
            tc::mma_f16(tm + TM_O, dvh, desc_at(dml, so), id16, true);
            tc::mma_f16(tm + TM_O, dvl, desc_at(dmh, so), id16, true);
            tc::mma_f16(tm + TM_S, dvh, desc_at(dkh, so), id128, true);
            tc::mma_f16(tm + TM_S, dvh, desc_at(dkl, so), id128, true);
            tc::mma_f16(tm + TM_S, dvl, desc_at(dkh, so), id128, true);
            tc::mma_commit(&ps.mma_bar);
        };
        if (lane == 0) {
            prefetch_tensormap(&tmz);
            for (int n = 0; n < NSTG && n < nchunk; ++n) issue(n);
        }
        cta_sync();  // S^T and its operand are in
        if (lane == 0) issue_p(0);
#pragma unroll 1
        for (int n = 0; n < nchunk; ++n) {
            cta_sync();  // V_new^T and the decayed S^T are in
            if (lane == 0) issue_o(n);
            cta_sync();  // the stage is consumed; the new S^T operand is in
            if (lane == 0) {
                if (n + NSTG < nchunk) issue(n + NSTG);
                if (n + 1 < nchunk) issue_p(n + 1);  // overlaps the norm and the stores
            }
        }
        if (!ok) ps.fail = 1;
    } else {
        // state S[i][j] -> TMEM S^T and its split operand; half 0 takes rows i < 64
        {
            const float *Sg = a.state_in + head * KD * KD;
            for (int i0 = 64 * half; i0 < 64 * half + 64; i0 += 16) {
                float v[16];
#pragma unroll
                for (int ii = 0; ii < 16; ++ii) v[ii] = Sg[(i0 + ii) * KD + ch];
                tc::tmem_st16(tc::taddr(tm, lb, TM_S + i0), v);
                tc::put_row8(st_hi, st_lo, tc::op_offset(ch, i0, KD), v);
                tc::put_row8(st_hi, st_lo, tc::op_offset(ch, i0 + 8, KD), v + 8);
            }
        }
        publish_smem();

        const float nw = a.norm_w[ch];
        uint32_t mma_ph = 0;
        auto mma_wait = [&]() {
            if (ok) ok = mbar_wait_bounded(&ps.mma_bar, mma_ph);
            mma_ph ^= 1u;
            tc::fence_after_sync();
        };

#pragma unroll 1
        for (int n = 0; n < nchunk; ++n) {
            const int t0 = n * KC, nt = min(KC, a.T - t0);
            const unsigned char *B = sm + (n % NSTG) * STAGE;
            if (ok) ok = mbar_wait_bounded(&ps.full[n % NSTG], static_cast<uint32_t>((n / NSTG) & 1));
            mma_wait();  // [P | Q']^T of this chunk

            // 2. V_new = U - P as the split operand V_new^T; S^T <- e^{G_last} S^T by state row
            if (half == 0) {
                float p[16];
                tc::tmem_ld16(tc::taddr(tm, lb, TM_P), p);
                const float *U = reinterpret_cast<const float *>(B + BW_U);
#pragma unroll
                for (int t = 0; t < KC; ++t) p[t] = U[t * KD + ch] - p[t];
                tc::put_row8(vn_hi, vn_lo, tc::op_offset(ch, 0, KC), p);
                tc::put_row8(vn_hi, vn_lo, tc::op_offset(ch, 8, KC), p + 8);
            }
            {
                const float *gl = reinterpret_cast<const float *>(B + BW_G);
                for (int i0 = 64 * half; i0 < 64 * half + 64; i0 += 16) {
                    float sv[16];
                    tc::tmem_ld16(tc::taddr(tm, lb, TM_S + i0), sv);
#pragma unroll
                    for (int ii = 0; ii < 16; ++ii) sv[ii] *= gl[i0 + ii];
                    tc::tmem_st16(tc::taddr(tm, lb, TM_S + i0), sv);
                }
            }
            publish_smem();
            mma_wait();  // O^T and the new S^T

            // 4. each half: o, its squares and the output gate of tokens 8 half .. +7, and
            // the new S^T of rows 64 half .. +63 as the next chunk's operand
            float o[8], gz[8];
            tc::tmem_ld8(tc::taddr(tm, lb, TM_O + 8 * half), o);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int t = 8 * half + j;
                sq[t * SQS + ch] = o[j] * o[j];
                const float zz = a.in_bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(B + STAGE_Z)[t * KD + ch])
                                           : reinterpret_cast<const float *>(B + STAGE_Z)[t * KD + ch];
                gz[j] = nw * (a.sig_gate ? fast_sigmoid(zz) : fast_silu(zz));
            }
            for (int i0 = 64 * half; i0 < 64 * half + 64; i0 += 16) {
                float sv[16];
                tc::tmem_ld16(tc::taddr(tm, lb, TM_S + i0), sv);
                tc::put_row8(st_hi, st_lo, tc::op_offset(ch, i0, KD), sv);
                tc::put_row8(st_hi, st_lo, tc::op_offset(ch, i0 + 8, KD), sv + 8);
            }
            publish_smem();  // the stage is consumed; o^2 and the S^T operand are in

            // 5. gated RMSNorm over the 128 columns of each token (16 threads a token)
            {
                const int t = tid >> 4, part = tid & 15;
                float s_ = 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) s_ += sq[t * SQS + 8 * part + j];
                s_ += __shfl_xor_sync(0xffffffffu, s_, 1);
                s_ += __shfl_xor_sync(0xffffffffu, s_, 2);
                s_ += __shfl_xor_sync(0xffffffffu, s_, 4);
                s_ += __shfl_xor_sync(0xffffffffu, s_, 8);
                if (part == 0) ps.rinv[t] = 1.0f / sqrtf(s_ / static_cast<float>(KD) + a.eps_norm);
            }
            compute_sync();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int t = 8 * half + j;
                if (t < nt) {
                    const size_t idx = ((static_cast<size_t>(b) * a.Ts + t0 + t) * a.H_v + h) * KD + ch;
                    const float yv = o[j] * ps.rinv[t] * gz[j];
                    if (a.out_bf16)
                        reinterpret_cast<__nv_bfloat16 *>(a.out)[idx] = __float2bfloat16_rn(yv);
                    else
                        reinterpret_cast<float *>(a.out)[idx] = yv;
                }
            }
        }

        // final state S[i][j] from S^T (lane j)
        {
            float *So = a.state_out + head * KD * KD;
            for (int i0 = 64 * half; i0 < 64 * half + 64; i0 += 16) {
                float sv[16];
                tc::tmem_ld16(tc::taddr(tm, lb, TM_S + i0), sv);
#pragma unroll
                for (int ii = 0; ii < 16; ++ii) So[(i0 + ii) * KD + ch] = sv[ii];
            }
        }
        // final conv window: rows T, T+1, T+2 of [kept window; the T new rows].  v
        // channels by their head, q and k channels by the group's first value head
        {
            const int hq = h / a.group;
            const size_t C = static_cast<size_t>(a.C);
            int chn[2], nc = 0;
            if (half == 0) {
                chn[nc++] = 2 * a.H_qk * KD + h * KD + ch;
            } else if (h % a.group == 0) {
                chn[nc++] = hq * KD + ch;
                chn[nc++] = a.H_qk * KD + hq * KD + ch;
            }
            for (int m = 0; m < nc; ++m) {
                const int c = chn[m];
                float x3[3];
#pragma unroll
                for (int j = 0; j < 3; ++j) {
                    const int idx = a.T + j;
                    x3[j] = idx < 3 ? a.conv_in[(static_cast<size_t>(b) * 3 + idx) * C + c]
                                    : ld_in(a.qkv, (static_cast<size_t>(b) * a.Ts + idx - 3) * C + c, a.in_bf16);
                }
#pragma unroll
                for (int j = 0; j < 3; ++j) a.conv_out[(static_cast<size_t>(b) * 3 + j) * C + c] = x3[j];
            }
        }
        if (!ok) ps.fail = 1;
    }
    cta_sync();
    if (ps.fail && tid == ISSUER_WARP * 32) {
        // a wait gave up: let the copies and products still in flight land
        // (bounded) before the shared memory and TMEM are released
        for (int s = 0; s < NSTG && s < nchunk; ++s) {
            const int last = s + NSTG * ((nchunk - 1 - s) / NSTG);
            mbar_wait_bounded(&ps.full[s], static_cast<uint32_t>((last / NSTG) & 1));
        }
        mbar_wait_bounded(&ps.mma_bar, static_cast<uint32_t>((2 * nchunk - 1) & 1));
        atomicOr(&g_kda_error, 1u);
    }
    tc::fence_before_sync();
    cta_sync();
    if (warp == 0) tc::tmem_dealloc(tm, TM_COLS);
}

}  // namespace

bool kda_chunk_shape(const gdn_shape_t &s)
{
    return s.d_k == KD && s.d_v == KD && s.T > 4 && s.conv_K == 4 &&
           static_cast<long long>(s.B) * s.T < (1LL << 31);
}

bool kda_chunk_pointers_ok(const StepArgs &a)
{
    // z goes by TMA; so do bf16 q/k/v rows and per-channel gate rows
    const auto al16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    return al16(a.z) && (!a.in_bf16 || (al16(a.qkv) && (!a.kda || al16(a.f))));
}

size_t kda_chunk_workspace_bytes(const gdn_shape_t &s)
{
    const size_t nchunk = (static_cast<size_t>(s.T) + KC - 1) / KC;
    return static_cast<size_t>(s.B) * s.H_v * nchunk * BLOCK_BYTES;
}

cudaError_t launch_kda_chunked(const StepArgs &a, void *workspace, cudaStream_t stream)
{
    static bool attr_set[64];  // per device; benign race: every writer sets the same value
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    constexpr int SMEM = SS_BYTES;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(kda_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (e != cudaSuccess) return e;
        // the intra kernel's rows exceed the 48 KB default; four CTAs an SM keep their share
        void (*intra[4])(StepArgs, unsigned char *, CUtensorMap, CUtensorMap) = {
            kda_intra_kernel<true, true>, kda_intra_kernel<true, false>,
            kda_intra_kernel<false, true>, kda_intra_kernel<false, false>};
        for (auto fn : intra) {
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, INTRA_SMEM);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
            if (e != cudaSuccess) return e;
        }
        attr_set[dev] = true;
    }
    const int nchunk = (a.T + KC - 1) / KC;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    CUtensorMap tmz;
    {   // z as [B*T][H_v][128] in the input dtype, boxes of 16 tokens x 1 head x 128 channels
        const uint64_t es = a.in_bf16 ? 2 : 4;
        const uint64_t dim[3] = {KD, static_cast<uint64_t>(a.H_v), static_cast<uint64_t>(a.B) * a.Ts};
        const uint64_t stride[2] = {KD * es, static_cast<uint64_t>(a.H_v) * KD * es};
        const uint32_t box[3] = {KD, 1, KC};
        if (!encode_tiled(&tmz, a.in_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                          a.z, dim, stride, box))
            return cudaErrorInvalidValue;
    }
    CUtensorMap tq = {}, tf = {};
    if (a.in_bf16) {
        {   // qkv as [B*T rows][C channels], boxes of 19 rows x 128 channels
            const uint64_t dim[2] = {static_cast<uint64_t>(a.C), static_cast<uint64_t>(a.B) * a.Ts};
            const uint64_t stride[1] = {static_cast<uint64_t>(a.C) * 2};
            const uint32_t box[2] = {KD, RAW_ROWS};
            if (!encode_tiled(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.qkv, dim, stride, box))
                return cudaErrorInvalidValue;
        }
        if (a.kda) {  // per-channel gate rows as [B*T][H_v][128], boxes of 16 tokens
            const uint64_t dim[3] = {KD, static_cast<uint64_t>(a.H_v), static_cast<uint64_t>(a.B) * a.Ts};
            const uint64_t stride[2] = {KD * 2, static_cast<uint64_t>(a.H_v) * KD * 2};
            const uint32_t box[3] = {KD, 1, KC};
            if (!encode_tiled(&tf, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.f, dim, stride, box))
                return cudaErrorInvalidValue;
        }
    }
    const dim3 grid(nchunk, a.H_v, a.B);
    if (a.in_bf16 && a.kda)
        kda_intra_kernel<true, true><<<grid, 256, INTRA_SMEM, stream>>>(a, ws, tq, tf);
    else if (a.in_bf16)
        kda_intra_kernel<true, false><<<grid, 256, INTRA_SMEM, stream>>>(a, ws, tq, tf);
    else if (a.kda)
        kda_intra_kernel<false, true><<<grid, 256, INTRA_SMEM, stream>>>(a, ws, tq, tf);
    else
        kda_intra_kernel<false, false><<<grid, 256, INTRA_SMEM, stream>>>(a, ws, tq, tf);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    kda_state_kernel<<<dim3(a.H_v, a.B), ST_THREADS, SMEM, stream>>>(a, ws, nchunk, tmz);
    return cudaGetLastError();
}

unsigned int take_kda_prefill_error()
{
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_kda_error, sizeof(v)) != cudaSuccess) return ~0u;
    if (v && cudaMemcpyToSymbol(g_kda_error, &zero, sizeof(zero)) != cudaSuccess) return ~0u;
    return v;
}

}  // namespace gdn
