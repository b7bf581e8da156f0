// Recurrent KDA / Gated DeltaNet step on sm_103a, persistent streaming form
// for many (sequence, value head) units with d_k = d_v = 128 and ungrouped
// heads: batched decode (T = 1) and verify (T <= 4).
//
// Two CTAs of 8 warps per SM; each walks the heads j = blockIdx.x,
// + gridDim.x, ...  Warp w owns state rows 16w..16w+15, one float4 of
// columns per lane.  Everything a head needs arrives by TMA bulk copies
// (cp.async.bulk, completing on mbarriers) into shared memory ahead of its
// turn:
//   * the 64 KiB fp32 state tile (contiguous): one stage per CTA, refilled
//     with the CTA's next head as soon as the current tile is in registers;
//   * the head's inputs and parameters (q/k/v rows, gate and output-gate
//     rows, beta, the conv window, conv weights, dt_bias, A_log): a ring of
//     IN_STAGES small stages, refilled with the head IN_STAGES positions ahead
//     once a head is finished.
// With the memory system saturated a single load waits several microseconds,
// so nothing on a head's critical path is fetched on demand; and with two
// CTAs per SM one CTA's stores overlap the other's arithmetic.  Per token:
// conv + gates on 256 threads, the decay pass with both column reductions in
// registers, a two-stage cross-warp reduction in shared memory, the gated
// RMSNorm on 128 threads, and 128-bit streaming stores of the new state
// straight from registers.
//
// Scalars (beta, A_log and, for per-head gates, f and dt_bias) come in the
// aligned 16-byte chunk that contains them; the host only selects this kernel
// when every such chunk lies inside its buffer (see stream_eligible).
#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

using namespace dev;

constexpr int SD = 128;                 // d_k = d_v
constexpr int KM1 = 3;                  // conv window rows
constexpr int IN_STAGES = 2;
constexpr int MAX_T = 4;
constexpr int CW = 8;                   // warps; warp w owns state rows 16w .. 16w+15
constexpr int NTHREADS = CW * 32;
constexpr int ROWS = SD / CW;
constexpr uint32_t TILE_BYTES = SD * SD * 4;

// Byte offsets of one input stage for T tokens of es-byte inputs.
struct InLayout {
    int qkv, win, cw, f, z, dt, beta, alog, bytes;
};

__host__ __device__ __forceinline__ InLayout in_layout(int T, int es, int kda)
{
    InLayout L;
    L.qkv = 0;                               // [T][3][SD] inputs
    L.win = L.qkv + T * 3 * SD * es;         // [3 rows][3][SD] fp32
    L.cw = L.win + KM1 * 3 * SD * 4;         // [3][SD] float4
    L.f = L.cw + 3 * SD * 16;                // [T][SD] inputs (per channel) or [T][16 B]
    L.z = L.f + T * (kda ? SD * es : 16);    // [T][SD] inputs
    L.dt = L.z + T * SD * es;                // [SD] fp32 or 16 B
    L.beta = L.dt + (kda ? SD * 4 : 16);     // [T][16 B]
    L.alog = L.beta + T * 16;                // 16 B
    L.bytes = (L.alog + 16 + 127) / 128 * 128;
    return L;
}

__device__ unsigned int g_stream_error;  // bit 0: a bounded mbarrier wait gave up

// The c-th TMA copy of head j's input bundle; false past the last one.
__device__ __forceinline__ bool input_copy(const StepArgs &a, const InLayout &L, int j, int c,
                                           const char *&src, int &dst, uint32_t &bytes)
{
    const int b = j / a.H_v, h = j % a.H_v;
    const int es = a.in_bf16 ? 2 : 4;
    const int T = a.T, C = a.C;
    const int ch[3] = {h * SD, a.H_qk * SD + h * SD, 2 * a.H_qk * SD + h * SD};
    if (c < 3 * T) {  // q, k, v rows of token t
        const int t = c / 3, sg = c % 3;
        src = static_cast<const char *>(a.qkv) + ((static_cast<size_t>(b) * T + t) * C + ch[sg]) * es;
        dst = L.qkv + (t * 3 + sg) * SD * es;
        bytes = SD * es;
        return true;
    }
    c -= 3 * T;
    if (c < 9) {  // conv window rows
        const int r = c / 3, sg = c % 3;
        src = reinterpret_cast<const char *>(a.conv_in + (static_cast<size_t>(b) * KM1 + r) * C + ch[sg]);
        dst = L.win + (r * 3 + sg) * SD * 4;
        bytes = SD * 4;
        return true;
    }
    c -= 9;
    if (c < 3) {  // conv weights of the head's q, k, v channels
        src = reinterpret_cast<const char *>(a.conv_w + static_cast<size_t>(ch[c]) * 4);
        dst = L.cw + c * SD * 16;
        bytes = SD * 16;
        return true;
    }
    c -= 3;
    if (c < 3 * T) {  // f, z, beta of token t
        const int t = c / 3, kind = c % 3;
        const size_t e = (static_cast<size_t>(b) * T + t) * a.H_v + h;
        if (kind == 0 && a.kda) {
            src = static_cast<const char *>(a.f) + e * SD * es;
            dst = L.f + t * SD * es;
            bytes = SD * es;
        } else if (kind == 0) {
            src = static_cast<const char *>(a.f) + ((e * es) & ~size_t(15));
            dst = L.f + t * 16;
            bytes = 16;
        } else if (kind == 1) {
            src = static_cast<const char *>(a.z) + e * SD * es;
            dst = L.z + t * SD * es;
            bytes = SD * es;
        } else {
            src = static_cast<const char *>(a.beta) + ((e * es) & ~size_t(15));
            dst = L.beta + t * 16;
            bytes = 16;
        }
        return true;
    }
    c -= 3 * T;
    if (c == 0) {  // dt_bias
        if (a.kda) {
            src = reinterpret_cast<const char *>(a.dt_bias + static_cast<size_t>(h) * SD);
            bytes = SD * 4;
        } else {
            src = reinterpret_cast<const char *>(a.dt_bias) + ((static_cast<size_t>(h) * 4) & ~size_t(15));
            bytes = 16;
        }
        dst = L.dt;
        return true;
    }
    if (c == 1) {  // A_log
        src = reinterpret_cast<const char *>(a.A_log) + ((static_cast<size_t>(h) * 4) & ~size_t(15));
        dst = L.alog;
        bytes = 16;
        return true;
    }
    return false;
}

__device__ __forceinline__ uint32_t input_bytes(const StepArgs &a)
{
    const uint32_t es = a.in_bf16 ? 2 : 4, T = a.T;
    return T * 3 * SD * es + 9 * SD * 4 + 3 * SD * 16 + T * (a.kda ? SD * es : 16) +
           T * SD * es + T * 16 + (a.kda ? SD * 4 : 16) + 16;
}

// Warp 0 queues head j's input bundle into `stage` (lane 0 arms the barrier first).
__device__ __forceinline__ void issue_inputs(const StepArgs &a, const InLayout &L, int j,
                                             char *stage, uint64_t *bar, int lane)
{
    if (lane == 0) mbar_expect_tx(bar, input_bytes(a));
    __syncwarp();
    for (int c = lane; c < 6 * a.T + 14; c += 32) {
        const char *src;
        int dst;
        uint32_t bytes;
        if (input_copy(a, L, j, c, src, dst, bytes)) tma_load_1d(stage + dst, src, bytes, bar);
    }
}

__device__ __forceinline__ float smem_in(const char *p, int idx, int bf16)
{
    if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[idx]);
    return reinterpret_cast<const float *>(p)[idx];
}

// Scalar element e of a buffer whose aligned 16-byte chunk sits at p.
__device__ __forceinline__ float chunk_in(const char *p, size_t e, int es)
{
    const int off = static_cast<int>((e * es) & 15);
    if (es == 2) return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(p + off));
    return *reinterpret_cast<const float *>(p + off);
}

struct Shared {
    float q[SD], k[SD], a[SD], v[SD], gz[SD], u[SD];
    float red3[4][3];
    float red_p[4];
    float red_k[CW][SD];
    float red_q[CW][SD];
    float beta;
    uint64_t tile_full;
    uint64_t in_full[IN_STAGES];
};

__global__ void __launch_bounds__(NTHREADS, 2) stream_kernel(const StepArgs a, int n_heads)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float *tile = reinterpret_cast<float *>(smem_raw);                 // [SD * SD]
    char *ins = reinterpret_cast<char *>(smem_raw) + TILE_BYTES;       // [IN_STAGES][L.bytes]
    __shared__ __align__(16) Shared sh;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = gridDim.x, c0 = blockIdx.x;
    const int C = a.C, es = a.in_bf16 ? 2 : 4;
    const InLayout L = in_layout(a.T, es, a.kda);
    const bool qk_thr = tid < SD;  // q_i, k_i of channel tid; threads SD..2SD-1: v, gate, z
    const int ch = tid & (SD - 1);
    const int row0 = ROWS * warp, col0 = 4 * lane;

    if (tid == 0) {
        mbar_init(&sh.tile_full, 1);
        for (int s = 0; s < IN_STAGES; ++s) mbar_init(&sh.in_full[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();
    // The state is not written by the previous kernel on the stream (launch
    // contract): the first tile is requested before the dependency wait.
    if (tid == 0) {
        mbar_expect_tx(&sh.tile_full, TILE_BYTES);
        tma_load_1d(tile, a.state_in + static_cast<size_t>(c0) * SD * SD, TILE_BYTES, &sh.tile_full);
    }
    const float nw = a.norm_w[ch];
    pdl_wait();  // inputs may be written by the previous kernel on the stream
    if (warp == 0) {
        for (int s = 0; s < IN_STAGES; ++s) {
            const int j = c0 + s * G;
            if (j < n_heads) issue_inputs(a, L, j, ins + s * L.bytes, &sh.in_full[s], lane);
        }
    }

    bool ok = true;
    int k = 0;
#pragma unroll 1
    for (int j = c0; j < n_heads; j += G, ++k) {
        const int is = k % IN_STAGES;
        const int b = j / a.H_v, h = j % a.H_v;
        char *in = ins + is * L.bytes;
        ok &= mbar_wait_bounded(&sh.in_full[is], static_cast<uint32_t>(k / IN_STAGES) & 1u);
        ok &= mbar_wait_bounded(&sh.tile_full, static_cast<uint32_t>(k) & 1u);

        // conv window, conv weights and gate parameters of this thread's channel
        const float *win = reinterpret_cast<const float *>(in + L.win);
        const float4 *cwv = reinterpret_cast<const float4 *>(in + L.cw);
        float w0[KM1], w1[KM1];
        float4 cw0, cw1 = make_float4(0.f, 0.f, 0.f, 0.f);
        float dtb = 0.f;
        if (qk_thr) {
#pragma unroll
            for (int r = 0; r < KM1; ++r) {
                w0[r] = win[(r * 3 + 0) * SD + ch];
                w1[r] = win[(r * 3 + 1) * SD + ch];
            }
            cw0 = cwv[ch];
            cw1 = cwv[SD + ch];
        } else {
#pragma unroll
            for (int r = 0; r < KM1; ++r) w0[r] = win[(r * 3 + 2) * SD + ch];
            cw0 = cwv[2 * SD + ch];
            if (a.kda) dtb = reinterpret_cast<const float *>(in + L.dt)[ch];
        }
        const float A = expf(chunk_in(in + L.alog, h, 4));
        const float dtb_head = a.kda ? 0.0f : chunk_in(in + L.dt, h, 4);

        float4 st[ROWS];
#pragma unroll
        for (int r = 0; r < ROWS; ++r)
            st[r] = *reinterpret_cast<const float4 *>(tile + (row0 + r) * SD + col0);

#pragma unroll 1
        for (int t = 0; t < a.T; ++t) {
            if (t > 0) __syncthreads();  // previous token's shared-memory reads are done
            const size_t e = (static_cast<size_t>(b) * a.T + t) * a.H_v + h;  // (b, t, h)
            const char *qkv = in + L.qkv + t * 3 * SD * es;

            // 1. conv + SiLU, L2-norm partial sums (q/k threads); v, decay and the
            //    output gate w * silu(z) (v threads)
            if (qk_thr) {
                const float xq = smem_in(qkv, ch, a.in_bf16);
                const float xk = smem_in(qkv, SD + ch, a.in_bf16);
                const float q = conv4_silu(cw0, w0, xq);
                const float kk = conv4_silu(cw1, w1, xk);
                w0[0] = w0[1]; w0[1] = w0[2]; w0[2] = xq;
                w1[0] = w1[1]; w1[1] = w1[2]; w1[2] = xk;
                sh.q[ch] = q;
                sh.k[ch] = kk;
                float sq = q * q, sk = kk * kk, sqk = q * kk;
                if (tid == 0) {
                    if (!a.kda)
                        sh.a[0] = expf(-A * softplus_f(chunk_in(in + L.f + t * 16, e, es) + dtb_head));
                    sh.beta = sigmoid_f(chunk_in(in + L.beta + t * 16, e, es));
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    sq += __shfl_xor_sync(0xffffffffu, sq, off);
                    sk += __shfl_xor_sync(0xffffffffu, sk, off);
                    sqk += __shfl_xor_sync(0xffffffffu, sqk, off);
                }
                if (lane == 0) {
                    sh.red3[warp][0] = sq;
                    sh.red3[warp][1] = sk;
                    sh.red3[warp][2] = sqk;
                }
            } else {
                const float xv = smem_in(qkv, 2 * SD + ch, a.in_bf16);
                sh.v[ch] = conv4_silu(cw0, w0, xv);
                w0[0] = w0[1]; w0[1] = w0[2]; w0[2] = xv;
                if (a.kda)
                    sh.a[ch] = expf(-A * softplus_f(smem_in(in + L.f + t * SD * es, ch, a.in_bf16) + dtb));
                sh.gz[ch] = nw * silu_f(smem_in(in + L.z + t * SD * es, ch, a.in_bf16));
            }
            __syncthreads();

            // the tile is in registers everywhere: bring in the CTA's next head
            if (t == 0 && tid == 0 && j + G < n_heads) {
                fence_proxy_async_smem();
                mbar_expect_tx(&sh.tile_full, TILE_BYTES);
                tma_load_1d(tile, a.state_in + static_cast<size_t>(j + G) * SD * SD, TILE_BYTES,
                            &sh.tile_full);
            }

            float Sq = 0.f, Sk = 0.f, Sqk = 0.f;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                Sq += sh.red3[w][0];
                Sk += sh.red3[w][1];
                Sqk += sh.red3[w][2];
            }
            const float rq = a.q_scale / sqrtf(Sq + a.eps_l2);
            const float rk = 1.0f / sqrtf(Sk + a.eps_l2);
            const float kq = Sqk * rq * rk;

            // 2. decay and the two column reductions over this warp's 16 rows
            float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
            for (int r4 = 0; r4 < ROWS / 4; ++r4) {
                const float4 k4 = *reinterpret_cast<const float4 *>(&sh.k[row0 + 4 * r4]);
                const float4 q4 = *reinterpret_cast<const float4 *>(&sh.q[row0 + 4 * r4]);
                float4 a4 = make_float4(sh.a[0], sh.a[0], sh.a[0], sh.a[0]);
                if (a.kda) a4 = *reinterpret_cast<const float4 *>(&sh.a[row0 + 4 * r4]);
                const float kv[4] = {k4.x, k4.y, k4.z, k4.w}, qv[4] = {q4.x, q4.y, q4.z, q4.w};
                const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = 4 * r4 + i;
                    const float al = av[i];
                    const float kr = kv[i] * rk, qr = qv[i] * rq;
                    st[r].x *= al; st[r].y *= al; st[r].z *= al; st[r].w *= al;
                    pk.x = fmaf(st[r].x, kr, pk.x); pk.y = fmaf(st[r].y, kr, pk.y);
                    pk.z = fmaf(st[r].z, kr, pk.z); pk.w = fmaf(st[r].w, kr, pk.w);
                    pq.x = fmaf(st[r].x, qr, pq.x); pq.y = fmaf(st[r].y, qr, pq.y);
                    pq.z = fmaf(st[r].z, qr, pq.z); pq.w = fmaf(st[r].w, qr, pq.w);
                }
            }
            *reinterpret_cast<float4 *>(&sh.red_k[warp][col0]) = pk;
            *reinterpret_cast<float4 *>(&sh.red_q[warp][col0]) = pq;
            __syncthreads();

            // 3. column sums, u and o for column ch; sum of o^2 per warp
            float o = 0.f;
            if (qk_thr) {
                float kS = 0.f, qS = 0.f;
#pragma unroll
                for (int w = 0; w < CW; ++w) {
                    kS += sh.red_k[w][ch];
                    qS += sh.red_q[w][ch];
                }
                const float u = sh.beta * (sh.v[ch] - kS);
                o = fmaf(kq, u, qS);
                sh.u[ch] = u;
                float p = o * o;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
                if (lane == 0) sh.red_p[warp] = p;
            }
            __syncthreads();

            // 4. gated RMSNorm output (column ch) and the state update
            if (qk_thr) {
                const float ss = sh.red_p[0] + sh.red_p[1] + sh.red_p[2] + sh.red_p[3];
                const float rinv = 1.0f / sqrtf(ss / static_cast<float>(SD) + a.eps_norm);
                const float y = o * rinv * sh.gz[ch];
                if (a.out_bf16)
                    reinterpret_cast<__nv_bfloat16 *>(a.out)[e * SD + ch] = __float2bfloat16_rn(y);
                else
                    reinterpret_cast<float *>(a.out)[e * SD + ch] = y;
            }
            const float4 u4 = *reinterpret_cast<const float4 *>(&sh.u[col0]);
#pragma unroll
            for (int r4 = 0; r4 < ROWS / 4; ++r4) {
                const float4 k4 = *reinterpret_cast<const float4 *>(&sh.k[row0 + 4 * r4]);
                const float kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = 4 * r4 + i;
                    const float kr = kv[i] * rk;
                    st[r].x = fmaf(kr, u4.x, st[r].x);
                    st[r].y = fmaf(kr, u4.y, st[r].y);
                    st[r].z = fmaf(kr, u4.z, st[r].z);
                    st[r].w = fmaf(kr, u4.w, st[r].w);
                }
            }
            float *dst = nullptr;
            if (a.state_hist)
                dst = a.state_hist + ((static_cast<size_t>(t) * a.B + b) * a.H_v + h) * SD * SD;
            else if (a.state_out && t == a.T - 1)
                dst = a.state_out + static_cast<size_t>(j) * SD * SD;
            if (dst) {
#pragma unroll
                for (int r = 0; r < ROWS; ++r)
                    __stcs(reinterpret_cast<float4 *>(dst + (row0 + r) * SD + col0), st[r]);
            }

            if (a.conv_hist) {
                float *chh = a.conv_hist + (static_cast<size_t>(t) * a.B + b) * KM1 * C;
                if (qk_thr) {
#pragma unroll
                    for (int r = 0; r < KM1; ++r) {
                        chh[static_cast<size_t>(r) * C + h * SD + ch] = w0[r];
                        chh[static_cast<size_t>(r) * C + a.H_qk * SD + h * SD + ch] = w1[r];
                    }
                } else {
#pragma unroll
                    for (int r = 0; r < KM1; ++r)
                        chh[static_cast<size_t>(r) * C + 2 * a.H_qk * SD + h * SD + ch] = w0[r];
                }
            }
        }

        if (a.conv_out) {
            float *co = a.conv_out + static_cast<size_t>(b) * KM1 * C;
            if (qk_thr) {
#pragma unroll
                for (int r = 0; r < KM1; ++r) {
                    co[static_cast<size_t>(r) * C + h * SD + ch] = w0[r];
                    co[static_cast<size_t>(r) * C + a.H_qk * SD + h * SD + ch] = w1[r];
                }
            } else {
#pragma unroll
                for (int r = 0; r < KM1; ++r)
                    co[static_cast<size_t>(r) * C + 2 * a.H_qk * SD + h * SD + ch] = w0[r];
            }
        }
        __syncthreads();  // this head's input stage and shared scratch are read out
        const int jr = j + IN_STAGES * G;
        if (warp == 0 && jr < n_heads) {
            if (lane == 0) fence_proxy_async_smem();
            __syncwarp();
            issue_inputs(a, L, jr, in, &sh.in_full[is], lane);
        }
    }
    if (!ok && lane == 0) atomicOr(&g_stream_error, 1u);
}

// 16-byte alignment of p and of the end of an n-byte buffer.
bool chunk_safe(const void *p, size_t n)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0 && (n & 15u) == 0;
}

}  // namespace

bool stream_eligible(const StepArgs &a)
{
    const size_t es = a.in_bf16 ? 2 : 4;
    const size_t bth = static_cast<size_t>(a.B) * a.T * a.H_v;
    bool ok = chunk_safe(a.qkv, static_cast<size_t>(a.C) * es) &&
              chunk_safe(a.z, SD * es) && chunk_safe(a.conv_in, static_cast<size_t>(a.C) * 4) &&
              chunk_safe(a.conv_w, 16) && chunk_safe(a.beta, bth * es) &&
              chunk_safe(a.A_log, static_cast<size_t>(a.H_v) * 4);
    if (a.kda)
        ok = ok && chunk_safe(a.f, SD * es) && chunk_safe(a.dt_bias, SD * 4);
    else
        ok = ok && chunk_safe(a.f, bth * es) && chunk_safe(a.dt_bias, static_cast<size_t>(a.H_v) * 4);
    return ok && a.T >= 1 && a.T <= MAX_T;
}

bool plan_stream(int D, int B, int H_v, int group, int num_sms, StepPlan *plan)
{
    const long units = static_cast<long>(B) * H_v;
    if (D != SD || group != 1 || units < 2L * num_sms || units > (1L << 30)) return false;
    plan->kind = StepPlan::kStream;
    plan->D = SD;
    plan->W = SD;
    plan->nslab = 1;
    plan->threads = NTHREADS;
    plan->cluster = 1;
    plan->grid = 2 * num_sms;
    plan->name = "stream<128>";
    return true;
}

cudaError_t launch_stream(const StepPlan &plan, const StepArgs &a, bool pdl, cudaStream_t stream)
{
    const int max_smem = TILE_BYTES + IN_STAGES * in_layout(MAX_T, 4, 1).bytes;
    static bool attr_set[64];  // per device; benign race: every writer sets the same value
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const InLayout L = in_layout(a.T, a.in_bf16 ? 2 : 4, a.kda);
    const int n_heads = a.B * a.H_v;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid < n_heads ? plan.grid : n_heads, 1, 1);
    cfg.blockDim = dim3(NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = TILE_BYTES + IN_STAGES * L.bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    int n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, stream_kernel, a, n_heads);
}

unsigned int take_stream_error()
{
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_stream_error, sizeof(v)) != cudaSuccess) return ~0u;
    if (v && cudaMemcpyToSymbol(g_stream_error, &zero, sizeof(zero)) != cudaSuccess) return ~0u;
    return v;
}

}  // namespace gdn
