// Chunked prefill for the per-channel decay (KDA), and for per-head decay shapes
// the tensor-core kernel does not take: two kernels over a device workspace.
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
// kda_intra_kernel: one CTA per (sequence, head, chunk), all chunks at once.  It
// runs the conv, the norms, the gates, the pair sums L and A and the forward
// substitution, and writes W, U, e^G * Q, e^{G_last - G} * K, A and e^{G_last}
// to the workspace (fp32).
// kda_state_kernel: one CTA per (sequence, head).  The fp32 state lives in
// registers; each chunk's block arrives by one TMA bulk copy into a ring of
// three stages; the products run as packed fp32 FMAs; the gated RMSNorm and the
// output store close each chunk.  The products are 16 x 128 x 128 per chunk: too
// thin for the tensor-core pipe's M = 64/128 tiles without a transposed state
// operand in shared memory, and fp32 keeps the state exact to rounding.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"
#include "gdn_device.cuh"
#include "gdn_internal.h"
#include "gdn_prefill.h"

namespace gdn {
namespace {

using namespace dev;

constexpr int KD = 128;  // d_k = d_v
constexpr int KC = 16;   // tokens per chunk
// Workspace block of one (sequence, head, chunk), in floats.  The three panels
// the state kernel reads by row quarters keep 4 spare floats after every 32
// channels, so the quarters of a row start in different shared-memory banks.
constexpr int KP = 144;
constexpr int OFF_W = 0;
constexpr int OFF_Q = KC * KP;
constexpr int OFF_K = 2 * KC * KP;
constexpr int OFF_U = 3 * KC * KP;
constexpr int OFF_A = OFF_U + KC * KD;
constexpr int OFF_G = OFF_A + KC * KC;
constexpr int BLOCK = OFF_G + KD;
constexpr uint32_t BLOCK_BYTES = BLOCK * 4;
static_assert(BLOCK_BYTES % 16 == 0, "bulk copies move multiples of 16 bytes");

__device__ unsigned int g_kda_error;

// position of channel r in a padded panel row
__host__ __device__ constexpr int pidx(int r) { return r + ((r >> 5) << 2); }

// Intra kernel staging rows: 136 floats, 4 spare after channel 63, so the two
// channel halves of a row sit in different banks.
constexpr int SP = 136;
__device__ __forceinline__ int hp(int i) { return i + ((i >> 6) << 2); }

// SiLU and sigmoid on the fast exponential and division: within a few units in
// the last place of fp32, far inside the prefill's tolerance.
__device__ __forceinline__ float fast_sigmoid(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }
__device__ __forceinline__ float fast_silu(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

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

__global__ void __launch_bounds__(256, 4) kda_intra_kernel(StepArgs a, float *ws)
{
    __shared__ __align__(16) float qs[KC][SP];
    __shared__ __align__(16) float ks[KC][SP];
    __shared__ __align__(16) float vs[KC][SP];
    __shared__ __align__(16) float gs[KC][SP];
    __shared__ __align__(16) float Ls[KC][KC];
    __shared__ __align__(16) float As[KC][KC];
    __shared__ float bs[KC];
    __shared__ float red[4][32];

    const int n = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int i = tid & (KD - 1);
    const int t0 = n * KC;
    const int nt = min(KC, a.T - t0);
    const int hq = h / a.group;
    const size_t C = static_cast<size_t>(a.C);
    const size_t row0 = static_cast<size_t>(b) * a.T + t0;

    // channel c's rows t0 - 3 .. t0 + 15: the three before t0 come from the
    // sequence, or from the kept window before its start; padded tokens read 0
    auto load_rows = [&](int c, float(&x)[KC + 3]) {
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const int tau = t0 - 3 + j;
            x[j] = tau >= 0 ? ld_in(a.qkv, (static_cast<size_t>(b) * a.T + tau) * C + c, a.in_bf16)
                            : a.conv_in[(static_cast<size_t>(b) * 3 + (3 + tau)) * C + c];
        }
#pragma unroll
        for (int t = 0; t < KC; ++t) x[3 + t] = t < nt ? ld_in(a.qkv, (row0 + t) * C + c, a.in_bf16) : 0.f;
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

    // ---- 1. conv, squares for the L2 norms, gates; padded tokens are zero
    if (tid < KC) bs[tid] = tid < nt ? fast_sigmoid(ld_in(a.beta, (row0 + tid) * a.H_v + h, a.in_bf16)) : 0.f;
    Ls[tid >> 4][tid & 15] = 0.f;
    As[tid >> 4][tid & 15] = 0.f;
    float q[KC], k[KC];
    if (tid < KD) {
        {
            const int cq = hq * KD + i, ck = a.H_qk * KD + hq * KD + i;
            float xq[KC + 3], xk[KC + 3];
            load_rows(cq, xq);
            load_rows(ck, xk);
            conv_rows(cq, xq, q);
            conv_rows(ck, xk, k);
        }
        float v[32];
#pragma unroll
        for (int t = 0; t < KC; ++t) {
            v[t] = q[t] * q[t];
            v[KC + t] = k[t] * k[t];
        }
        red[warp][lane] = reduce_scatter32(v, lane);
    } else {
        const int cv = 2 * a.H_qk * KD + h * KD + i;
        float xv[KC + 3], fl[KC];
        load_rows(cv, xv);
#pragma unroll
        for (int t = 0; t < KC; ++t) {
            const size_t bth = (row0 + t) * a.H_v + h;
            fl[t] = t < nt ? (a.kda ? ld_in(a.f, bth * KD + i, a.in_bf16) : ld_in(a.f, bth, a.in_bf16)) : 0.f;
        }
        float v[KC];
        conv_rows(cv, xv, v);
#pragma unroll
        for (int t = 0; t < KC; ++t) vs[t][hp(i)] = v[t];
        // log-decays of channel i summed along the chunk.  Softplus gates:
        // g = -exp(A_log) softplus(f + dt_bias); lower-bound gate: g = lb sigmoid(-a f)
        const float A = a.lb_gate ? a.A_log[h] : expf(a.A_log[h]);
        const float lbv = a.lb_gate ? a.dt_bias[h] : 0.f;
        const float dtb = a.lb_gate ? 0.f : (a.kda ? a.dt_bias[static_cast<size_t>(h) * KD + i] : a.dt_bias[h]);
        float G = 0.f;
#pragma unroll
        for (int t = 0; t < KC; ++t) {
            if (t < nt) G += a.lb_gate ? lbv * fast_sigmoid(-A * fl[t]) : -A * softplus_f(fl[t] + dtb);
            gs[t][hp(i)] = G;
        }
    }
    __syncthreads();
    if (tid < KD) {
#pragma unroll
        for (int t = 0; t < KC; ++t) {
            const float sq = red[0][t] + red[1][t] + red[2][t] + red[3][t];
            const float sk = red[0][KC + t] + red[1][KC + t] + red[2][KC + t] + red[3][KC + t];
            qs[t][hp(i)] = q[t] * (a.q_scale / sqrtf(sq + a.eps_l2));
            ks[t][hp(i)] = k[t] * (1.0f / sqrtf(sk + a.eps_l2));
        }
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
#pragma unroll 4
            for (int m = 0; m < 64; m += 4) {
                const float4 g1 = *reinterpret_cast<const float4 *>(&gs[t][base + m]);
                const float4 g0 = *reinterpret_cast<const float4 *>(&gs[s][base + m]);
                const float4 k1 = *reinterpret_cast<const float4 *>(&ks[t][base + m]);
                const float4 k0 = *reinterpret_cast<const float4 *>(&ks[s][base + m]);
                const float4 q1 = *reinterpret_cast<const float4 *>(&qs[t][base + m]);
                float e = __expf(g1.x - g0.x);
                kk = fmaf(k1.x * k0.x, e, kk);
                qk = fmaf(q1.x * k0.x, e, qk);
                e = __expf(g1.y - g0.y);
                kk = fmaf(k1.y * k0.y, e, kk);
                qk = fmaf(q1.y * k0.y, e, qk);
                e = __expf(g1.z - g0.z);
                kk = fmaf(k1.z * k0.z, e, kk);
                qk = fmaf(q1.z * k0.z, e, qk);
                e = __expf(g1.w - g0.w);
                kk = fmaf(k1.w * k0.w, e, kk);
                qk = fmaf(q1.w * k0.w, e, qk);
            }
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
                Ls[t][s] = bs[t] * (kk + kk2);
                As[t][s] = qk + qk2;
            }
        } else {
            As[t][t] = qk;
        }
    }
    __syncthreads();

    // ---- 3. (I + L) X = B by forward substitution, one column a thread:
    // W's columns from beta e^G k, U's from beta v; then the state stage's operands
    float *blk = ws + ((static_cast<size_t>(b) * a.H_v + h) * gridDim.x + n) * BLOCK;
    {
        const bool wside = tid < KD;
        float x[KC];
#pragma unroll
        for (int t = 0; t < KC; ++t)
            x[t] = bs[t] * (wside ? ks[t][hp(i)] * __expf(gs[t][hp(i)]) : vs[t][hp(i)]);
#pragma unroll
        for (int t = 1; t < KC; ++t)
#pragma unroll
            for (int s = 0; s < t; ++s) x[t] = fmaf(-Ls[t][s], x[s], x[t]);
        if (wside) {
#pragma unroll
            for (int t = 0; t < KC; ++t) {
                blk[OFF_W + t * KP + pidx(i)] = x[t];
                blk[OFF_Q + t * KP + pidx(i)] = qs[t][hp(i)] * __expf(gs[t][hp(i)]);
            }
        } else {
            const float Gl = gs[KC - 1][hp(i)];
#pragma unroll
            for (int t = 0; t < KC; ++t) {
                blk[OFF_U + t * KD + i] = x[t];
                blk[OFF_K + t * KP + pidx(i)] = ks[t][hp(i)] * __expf(Gl - gs[t][hp(i)]);
            }
            blk[OFF_G + i] = __expf(Gl);
        }
        blk[OFF_A + tid] = As[tid >> 4][tid & 15];
    }
}

// ---------------------------------------------------------------- state stage

constexpr int NSTG = 3;

struct StateSmem {
    float blk[NSTG][BLOCK];
    float red[2][8][KC];  // per warp, per token: partial sums of o^2, by chunk parity
    uint64_t full[NSTG];
};

__device__ __forceinline__ float2 lo2(const float4 v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 hi2(const float4 v) { return make_float2(v.z, v.w); }

__device__ __forceinline__ void store_out2(void *out, size_t idx, int bf16, float a, float b)
{
    if (bf16) {
        *reinterpret_cast<__nv_bfloat162 *>(reinterpret_cast<__nv_bfloat16 *>(out) + idx) =
            __floats2bfloat162_rn(a, b);
    } else {
        *reinterpret_cast<float2 *>(reinterpret_cast<float *>(out) + idx) = make_float2(a, b);
    }
}

// Thread layout: lane = row quarter rq (rows 32 rq .. 32 rq + 31) + 4 x column
// pair; warp w holds column pairs 8w .. 8w + 7, so a quad of lanes covers two
// full columns and the sums over rows are two shuffles.
__global__ void __launch_bounds__(256, 1) kda_state_kernel(StepArgs a, const float *ws, int nchunk)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    StateSmem &sm = *reinterpret_cast<StateSmem *>(smem_raw);
    const int h = blockIdx.x, b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rq = lane & 3;
    const int c0 = 2 * (warp * 8 + (lane >> 2));
    const size_t head = static_cast<size_t>(b) * a.H_v + h;
    const float *blocks = ws + head * nchunk * BLOCK;

    if (tid == 0) {
        for (int s = 0; s < NSTG; ++s) mbar_init(&sm.full[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        for (int s = 0; s < NSTG && s < nchunk; ++s) {
            mbar_expect_tx(&sm.full[s], BLOCK_BYTES);
            tma_load_1d(sm.blk[s], blocks + static_cast<size_t>(s) * BLOCK, BLOCK_BYTES, &sm.full[s]);
        }
    }

    // state rows 32 rq + 2p, +1 of columns c0 (sc0) and c0 + 1 (sc1), as row pairs
    float2 sc0[16], sc1[16];
    {
        const float *S = a.state_in + head * KD * KD + c0;
#pragma unroll
        for (int p = 0; p < 16; ++p) {
            const int r = 32 * rq + 2 * p;
            const float2 x = *reinterpret_cast<const float2 *>(S + static_cast<size_t>(r) * KD);
            const float2 y = *reinterpret_cast<const float2 *>(S + static_cast<size_t>(r + 1) * KD);
            sc0[p] = make_float2(x.x, y.x);
            sc1[p] = make_float2(x.y, y.y);
        }
    }
    const float nw0 = a.norm_w[c0], nw1 = a.norm_w[c0 + 1];
    bool ok = true;

#pragma unroll 1
    for (int n = 0; n < nchunk; ++n) {
        const int st = n % NSTG;
        const int t0 = n * KC, nt = min(KC, a.T - t0);
        // output-gate inputs of this lane's tokens 4 rq .. 4 rq + 3, issued early
        float z0[4], z1[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int t = 4 * rq + j;
            z0[j] = z1[j] = 0.f;
            if (t < nt) {
                const size_t idx = ((static_cast<size_t>(b) * a.T + t0 + t) * a.H_v + h) * KD + c0;
                z0[j] = ld_in(a.z, idx, a.in_bf16);
                z1[j] = ld_in(a.z, idx + 1, a.in_bf16);
            }
        }
        if (!mbar_wait_bounded(&sm.full[st], static_cast<uint32_t>((n / NSTG) & 1))) ok = false;
        const float *B = sm.blk[st];

        // 1. P = W S0 and Q' = (e^G Q) S0.  Tokens go in groups {j, j+4, j+8, j+12}
        // (16 independent accumulator chains), each group summed over the quad at
        // once so that lane rq keeps token j + 4 rq.  pv[0..3][j]: P col c0,
        // P col c0+1, Q' col c0, Q' col c0+1 of token 4 rq + j
        float pv[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float2 acc[4][4];
#pragma unroll
            for (int g = 0; g < 4; ++g)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[g][c] = make_float2(0.f, 0.f);
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                float4 w4[4], q4[4];
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const int t = j + 4 * g;
                    w4[g] = *reinterpret_cast<const float4 *>(B + OFF_W + t * KP + 36 * rq + 4 * m);
                    q4[g] = *reinterpret_cast<const float4 *>(B + OFF_Q + t * KP + 36 * rq + 4 * m);
                }
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    acc[g][0] = __ffma2_rn(lo2(w4[g]), sc0[2 * m], acc[g][0]);
                    acc[g][1] = __ffma2_rn(lo2(w4[g]), sc1[2 * m], acc[g][1]);
                    acc[g][2] = __ffma2_rn(lo2(q4[g]), sc0[2 * m], acc[g][2]);
                    acc[g][3] = __ffma2_rn(lo2(q4[g]), sc1[2 * m], acc[g][3]);
                }
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    acc[g][0] = __ffma2_rn(hi2(w4[g]), sc0[2 * m + 1], acc[g][0]);
                    acc[g][1] = __ffma2_rn(hi2(w4[g]), sc1[2 * m + 1], acc[g][1]);
                    acc[g][2] = __ffma2_rn(hi2(q4[g]), sc0[2 * m + 1], acc[g][2]);
                    acc[g][3] = __ffma2_rn(hi2(q4[g]), sc1[2 * m + 1], acc[g][3]);
                }
            }
            float r[4][4];
#pragma unroll
            for (int g = 0; g < 4; ++g)
#pragma unroll
                for (int c = 0; c < 4; ++c) r[g][c] = acc[g][c].x + acc[g][c].y;
            // xor 2: lanes with rq & 2 keep tokens g = 2, 3, the others g = 0, 1
            const bool up2 = (rq & 2) != 0;
#pragma unroll
            for (int g = 0; g < 2; ++g)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float send = up2 ? r[g][c] : r[g + 2][c];
                    const float keep = up2 ? r[g + 2][c] : r[g][c];
                    r[g][c] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
                }
            // xor 1: lanes with rq & 1 keep the odd one: g = rq
            const bool up1 = (rq & 1) != 0;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float send = up1 ? r[0][c] : r[1][c];
                const float keep = up1 ? r[1][c] : r[0][c];
                pv[c][j] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
            }
        }

        // 2. V_new = U - P for this lane's tokens, then gathered for all 16
        float V0[KC], V1[KC];
        {
            float vn0[4], vn1[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 u = *reinterpret_cast<const float2 *>(B + OFF_U + (4 * rq + j) * KD + c0);
                vn0[j] = u.x - pv[0][j];
                vn1[j] = u.y - pv[1][j];
            }
            float a0[8], a1[8];
            const bool up1 = (rq & 1) != 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float r0 = __shfl_xor_sync(0xffffffffu, vn0[j], 1);
                const float r1 = __shfl_xor_sync(0xffffffffu, vn1[j], 1);
                a0[j] = up1 ? r0 : vn0[j];
                a0[j + 4] = up1 ? vn0[j] : r0;
                a1[j] = up1 ? r1 : vn1[j];
                a1[j + 4] = up1 ? vn1[j] : r1;
            }
            const bool up2 = (rq & 2) != 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float r0 = __shfl_xor_sync(0xffffffffu, a0[j], 2);
                const float r1 = __shfl_xor_sync(0xffffffffu, a1[j], 2);
                V0[j] = up2 ? r0 : a0[j];
                V0[j + 8] = up2 ? a0[j] : r0;
                V1[j] = up2 ? r1 : a1[j];
                V1[j + 8] = up2 ? a1[j] : r1;
            }
        }

        // 3. O = Q' + A V_new (A is zero above the diagonal)
        float o0[4], o1[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 *ar = reinterpret_cast<const float4 *>(B + OFF_A + (4 * rq + j) * KC);
            float x0 = pv[2][j], x1 = pv[3][j];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float4 av = ar[m];
                x0 = fmaf(av.x, V0[4 * m], x0);
                x1 = fmaf(av.x, V1[4 * m], x1);
                x0 = fmaf(av.y, V0[4 * m + 1], x0);
                x1 = fmaf(av.y, V1[4 * m + 1], x1);
                x0 = fmaf(av.z, V0[4 * m + 2], x0);
                x1 = fmaf(av.z, V1[4 * m + 2], x1);
                x0 = fmaf(av.w, V0[4 * m + 3], x0);
                x1 = fmaf(av.w, V1[4 * m + 3], x1);
            }
            o0[j] = x0;
            o1[j] = x1;
        }

        // 4. S = Diag(e^{G_last}) S0 + Kd^T V_new
        {
            const float4 *gl = reinterpret_cast<const float4 *>(B + OFF_G + 32 * rq);
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const float4 g4 = gl[m];
                sc0[2 * m] = __fmul2_rn(sc0[2 * m], lo2(g4));
                sc0[2 * m + 1] = __fmul2_rn(sc0[2 * m + 1], hi2(g4));
                sc1[2 * m] = __fmul2_rn(sc1[2 * m], lo2(g4));
                sc1[2 * m + 1] = __fmul2_rn(sc1[2 * m + 1], hi2(g4));
            }
#pragma unroll
            for (int t = 0; t < KC; ++t) {
                const float4 *kr = reinterpret_cast<const float4 *>(B + OFF_K + t * KP + 36 * rq);
                const float2 v0 = make_float2(V0[t], V0[t]), v1 = make_float2(V1[t], V1[t]);
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const float4 k4 = kr[m];
                    sc0[2 * m] = __ffma2_rn(lo2(k4), v0, sc0[2 * m]);
                    sc0[2 * m + 1] = __ffma2_rn(hi2(k4), v0, sc0[2 * m + 1]);
                    sc1[2 * m] = __ffma2_rn(lo2(k4), v1, sc1[2 * m]);
                    sc1[2 * m + 1] = __ffma2_rn(hi2(k4), v1, sc1[2 * m + 1]);
                }
            }
        }

        // 5. gated RMSNorm over the head's 128 columns
        float ss[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) ss[j] = fmaf(o0[j], o0[j], o1[j] * o1[j]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1)
#pragma unroll
            for (int j = 0; j < 4; ++j) ss[j] += __shfl_xor_sync(0xffffffffu, ss[j], off);
        float(*rd)[KC] = sm.red[n & 1];
        if ((lane >> 2) == 0)
            *reinterpret_cast<float4 *>(&rd[warp][4 * rq]) = make_float4(ss[0], ss[1], ss[2], ss[3]);
        __syncthreads();  // the stage is consumed and the partial sums are in
        if (tid == 0 && n + NSTG < nchunk) {
            mbar_expect_tx(&sm.full[st], BLOCK_BYTES);
            tma_load_1d(sm.blk[st], blocks + static_cast<size_t>(n + NSTG) * BLOCK, BLOCK_BYTES,
                        &sm.full[st]);
        }
        float4 tot = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            const float4 r4 = *reinterpret_cast<const float4 *>(&rd[w][4 * rq]);
            tot.x += r4.x;
            tot.y += r4.y;
            tot.z += r4.z;
            tot.w += r4.w;
        }
        const float tv[4] = {tot.x, tot.y, tot.z, tot.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int t = 4 * rq + j;
            if (t < nt) {
                const float rinv = 1.0f / sqrtf(tv[j] / static_cast<float>(KD) + a.eps_norm);
                const float g0 = a.sig_gate ? sigmoid_f(z0[j]) : silu_f(z0[j]);
                const float g1 = a.sig_gate ? sigmoid_f(z1[j]) : silu_f(z1[j]);
                const size_t idx = ((static_cast<size_t>(b) * a.T + t0 + t) * a.H_v + h) * KD + c0;
                store_out2(a.out, idx, a.out_bf16, o0[j] * rinv * nw0 * g0, o1[j] * rinv * nw1 * g1);
            }
        }
    }
    if (!ok) atomicOr(&g_kda_error, 1u);

    // final state
    {
        float *So = a.state_out + head * KD * KD + c0;
#pragma unroll
        for (int p = 0; p < 16; ++p) {
            const int r = 32 * rq + 2 * p;
            *reinterpret_cast<float2 *>(So + static_cast<size_t>(r) * KD) = make_float2(sc0[p].x, sc1[p].x);
            *reinterpret_cast<float2 *>(So + static_cast<size_t>(r + 1) * KD) =
                make_float2(sc0[p].y, sc1[p].y);
        }
    }
    // final conv window: rows T, T+1, T+2 of [kept window; the T new rows].  v
    // channels by their head, q and k channels by the group's first value head
    {
        const int i = tid & (KD - 1);
        const int hq = h / a.group;
        const size_t C = static_cast<size_t>(a.C);
        int ch[2], nc = 0;
        if (tid < KD) {
            ch[nc++] = 2 * a.H_qk * KD + h * KD + i;
        } else if (h % a.group == 0) {
            ch[nc++] = hq * KD + i;
            ch[nc++] = a.H_qk * KD + hq * KD + i;
        }
        for (int m = 0; m < nc; ++m) {
            const int c = ch[m];
            float x[3];
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                const int idx = a.T + j;
                x[j] = idx < 3 ? a.conv_in[(static_cast<size_t>(b) * 3 + idx) * C + c]
                               : ld_in(a.qkv, (static_cast<size_t>(b) * a.T + idx - 3) * C + c, a.in_bf16);
            }
#pragma unroll
            for (int j = 0; j < 3; ++j) a.conv_out[(static_cast<size_t>(b) * 3 + j) * C + c] = x[j];
        }
    }
}

}  // namespace

bool kda_chunk_shape(const gdn_shape_t &s)
{
    return s.d_k == KD && s.d_v == KD && s.T > 4 && s.conv_K == 4 &&
           static_cast<long long>(s.B) * s.T < (1LL << 31);
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
    constexpr int SMEM = static_cast<int>(sizeof(StateSmem));
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(kda_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const int nchunk = (a.T + KC - 1) / KC;
    float *ws = static_cast<float *>(workspace);
    kda_intra_kernel<<<dim3(nchunk, a.H_v, a.B), 256, 0, stream>>>(a, ws);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    kda_state_kernel<<<dim3(a.H_v, a.B), 256, SMEM, stream>>>(a, ws, nchunk);
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
