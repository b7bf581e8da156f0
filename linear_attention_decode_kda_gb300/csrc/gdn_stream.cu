// Recurrent KDA / Gated DeltaNet step on sm_103a, persistent streaming form
// for many (sequence, value head) units with d_k = d_v = 128 and ungrouped
// heads: batched decode (T = 1) and verify (T <= 4).
//
// Two CTAs of 8 warps per SM; each walks the heads j = blockIdx.x,
// + gridDim.x, ...  Warp w owns state rows 16w..16w+15, one float4 of
// columns per lane.  Everything a head needs arrives by TMA into shared
// memory ahead of its turn, completing on mbarriers:
//   * the 64 KiB fp32 state tile (one bulk copy): one stage per CTA, refilled
//     with the CTA's next head as soon as the current tile is in registers;
//   * the head's inputs and parameters in ten copies -- q/k/v rows, conv
//     window, gate rows, output-gate rows and beta through tensor maps (each
//     copy spans all T tokens or all three q/k/v segments), the three 2 KiB
//     runs of conv weights, dt_bias and A_log as bulk copies -- into a ring of
//     input stages, each refilled as soon as its head's last token has read it.
// With the memory system saturated a single load waits several microseconds,
// so nothing on a head's critical path is fetched on demand; and with two
// CTAs per SM one CTA's stores overlap the other's arithmetic.
//
// Per head:
//   A. for each of its T tokens: conv + SiLU of q, k (threads 0..127) and of v
//      with the decay and the output gate w * silu(z) (threads 128..255), and
//      the L2-norm partial sums -- none of it depends on the state, so the T
//      tokens share one block barrier;
//   then per token, one block barrier: the decay pass over the warp's rows with
//   both column reductions (St^T k, St^T q) in registers, partials to shared
//   memory.  After it every warp sums the eight partials of its lanes' columns
//   itself, so u = beta (v - St^T k), o = St^T q + (k.q) u and the sum of o^2
//   over the head are known in every warp without a further barrier; one warp
//   writes the gated RMSNorm output, all warps update their rows and store them
//   with 128-bit streaming stores.
#include <cuda.h>

#include "gdn_device.cuh"
#include "gdn_internal.h"
#include "gdn_tmap.h"

namespace gdn {
namespace {

using namespace dev;

constexpr int SD = 128;                 // d_k = d_v
constexpr int KM1 = 3;                  // conv window rows
constexpr int MAX_STAGES = 2;           // input stages (1 when two do not fit)
constexpr int MAX_T = 4;
constexpr int CW = 8;                   // warps; warp w owns state rows 16w .. 16w+15
constexpr int NTHREADS = CW * 32;
constexpr int ROWS = SD / CW;
constexpr uint32_t TILE_BYTES = SD * SD * 4;
constexpr int SMEM_PER_SM = 228 * 1024;  // shared memory per SM, 1 KiB of it reserved per CTA

__host__ __device__ constexpr int up128(int x) { return (x + 127) / 128 * 128; }

// Byte offsets of one input stage for T tokens of es-byte inputs.
struct InLayout {
    int qkv, win, cw, f, z, beta, dt, alog, bytes;
};

// kda: gate rows per key channel; dtpc: dt_bias per key channel (the softplus KDA gate)
__host__ __device__ __forceinline__ InLayout in_layout(int T, int es, int kda, int dtpc)
{
    InLayout L;
    L.qkv = 0;                                      // [T][3][SD] inputs
    L.win = L.qkv + up128(T * 3 * SD * es);         // [3 rows][3][SD] fp32
    L.cw = L.win + up128(KM1 * 3 * SD * 4);         // [3][SD] float4
    L.f = L.cw + up128(3 * SD * 16);                // [T][SD] inputs, or [T][16 B] per head
    L.z = L.f + up128(T * (kda ? SD * es : 16));    // [T][SD] inputs
    L.beta = L.z + up128(T * SD * es);              // [T][16 B]
    L.dt = L.beta + up128(T * 16);                  // [SD] fp32, or 16 B
    L.alog = L.dt + up128(dtpc ? SD * 4 : 16);      // 16 B
    L.bytes = L.alog + 128;
    return L;
}

__host__ __device__ __forceinline__ uint32_t input_bytes(int T, int es, int kda, int dtpc)
{
    return T * 3 * SD * es + KM1 * 3 * SD * 4 + 3 * SD * 16 + T * (kda ? SD * es : 16) +
           T * SD * es + T * 16 + (dtpc ? SD * 4 : 16) + 16;
}

__host__ __device__ __forceinline__ int dt_per_channel(const StepArgs &a) { return a.kda && !a.lb_gate; }

// The tensor maps of the input bundle (kernel parameters).
struct InMaps {
    CUtensorMap qkv;   // {SD*H, 3, B*T}: box {SD, 3, T} -> q, k, v rows of T tokens
    CUtensorMap win;   // {SD*H, 3, B*3}: box {SD, 3, 3} -> the head's conv window
    CUtensorMap f;     // per channel {SD, H, B*T} box {SD, 1, T}; per head {H, B*T} box {16/es, T}
    CUtensorMap z;     // {SD, H, B*T}:   box {SD, 1, T}
    CUtensorMap beta;  // {H, B*T}:       box {16/es, T}
};

// Shared scratch.  Per-token rows are indexed by slot: token t of a
// multi-token head, or the head's parity when heads have one token.  The column
// partial sums (red_k, red_q) follow the input stages in dynamic shared memory:
// two buffers when a head has several tokens (token t+1's partials are written
// while slower warps may still read token t's), else one.
struct Shared {  // float4-read arrays first: every one starts on a 16-byte boundary
    __align__(16) float q[MAX_T][SD];
    __align__(16) float k[MAX_T][SD];
    __align__(16) float a[MAX_T][SD];
    __align__(16) float v[MAX_T][SD];
    __align__(16) float gz[MAX_T][SD];
    float red3[MAX_T][4][3];
    float beta[MAX_T];
    uint64_t tile_full;
    uint64_t in_full[MAX_STAGES];
};

constexpr int SH_BYTES = up128(static_cast<int>(sizeof(Shared)));

__host__ __device__ constexpr int n_red(int T) { return T > 1 ? 2 : 1; }

__device__ unsigned int g_stream_error;  // bit 0: a bounded mbarrier wait gave up

// Warp 0 queues head j's input bundle into `stage` (lane 0 arms the barrier first).
__device__ __forceinline__ void issue_inputs(const StepArgs &a, const InMaps &m, const InLayout &L,
                                             int j, char *stage, uint64_t *bar, int lane)
{
    const int b = j / a.H_v, h = j % a.H_v;
    const int es = a.in_bf16 ? 2 : 4, per16 = 16 / es;
    if (lane == 0) mbar_expect_tx(bar, input_bytes(a.T, es, a.kda, dt_per_channel(a)));
    __syncwarp();
    const int bt = b * a.T;
    switch (lane) {
    case 0: tma_load_3d(stage + L.qkv, &m.qkv, h * SD, 0, bt, bar); break;
    case 1: tma_load_3d(stage + L.win, &m.win, h * SD, 0, b * KM1, bar); break;
    case 2:  // conv weights of the head's q, k and v channels: 2 KiB contiguous each
        for (int sg = 0; sg < 3; ++sg)
            tma_load_1d(stage + L.cw + sg * SD * 16,
                        a.conv_w + (static_cast<size_t>(sg) * a.H_qk * SD + static_cast<size_t>(h) * SD) * 4,
                        SD * 16, bar);
        break;
    case 3:
        if (a.kda) tma_load_3d(stage + L.f, &m.f, 0, h, bt, bar);
        else tma_load_2d(stage + L.f, &m.f, h & ~(per16 - 1), bt, bar);
        break;
    case 4: tma_load_3d(stage + L.z, &m.z, 0, h, bt, bar); break;
    case 5: tma_load_2d(stage + L.beta, &m.beta, h & ~(per16 - 1), bt, bar); break;
    case 6:
        if (dt_per_channel(a)) tma_load_1d(stage + L.dt, a.dt_bias + static_cast<size_t>(h) * SD, SD * 4, bar);
        else tma_load_1d(stage + L.dt, a.dt_bias + (h & ~3), 16, bar);
        break;
    case 7: tma_load_1d(stage + L.alog, a.A_log + (h & ~3), 16, bar); break;
    default: break;
    }
}

__device__ __forceinline__ float smem_in(const char *p, int idx, int bf16)
{
    if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[idx]);
    return reinterpret_cast<const float *>(p)[idx];
}

__global__ void __launch_bounds__(NTHREADS, 2)
stream_kernel(const StepArgs a, const __grid_constant__ InMaps maps, int n_heads, int nst)
{
    extern __shared__ unsigned char smem_raw[];
    // 128-byte aligned base (TMA destinations)
    unsigned char *base = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);
    Shared &sh = *reinterpret_cast<Shared *>(base);
    float *tile = reinterpret_cast<float *>(base + SH_BYTES);            // [SD][SD]
    char *ins = reinterpret_cast<char *>(base + SH_BYTES + TILE_BYTES);  // [nst][L.bytes]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = gridDim.x, c0 = blockIdx.x;
    const int C = a.C, T = a.T, es = a.in_bf16 ? 2 : 4, per16 = 16 / es;
    const InLayout L = in_layout(T, es, a.kda, dt_per_channel(a));
    float *red = reinterpret_cast<float *>(ins + nst * L.bytes);  // [n_red][2][CW][SD]
    const bool qk_thr = tid < SD;  // q_i, k_i of channel tid; threads SD..2SD-1: gate, v, z
    const int ch = tid & (SD - 1);
    const int row0 = ROWS * warp, col0 = 4 * lane;

    if (tid == 0) {
        mbar_init(&sh.tile_full, 1);
        for (int s = 0; s < nst; ++s) mbar_init(&sh.in_full[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    // The state is not written by the previous kernel on the stream (launch
    // contract): the first tile is requested before the dependency wait.
    if (tid == 0) {
        mbar_expect_tx(&sh.tile_full, TILE_BYTES);
        tma_load_1d(tile, a.state_in + static_cast<size_t>(c0) * SD * SD, TILE_BYTES, &sh.tile_full);
    }
    const float nw = qk_thr ? 0.0f : a.norm_w[ch];
    if (tid == 0) {  // the input maps' descriptors, ahead of their first use
        prefetch_tensormap(&maps.qkv);
        prefetch_tensormap(&maps.win);
        prefetch_tensormap(&maps.f);
        prefetch_tensormap(&maps.z);
        prefetch_tensormap(&maps.beta);
    }
    pdl_wait();  // inputs may be written by the previous kernel on the stream
    // Dependents launch only once this grid has passed its own dependency wait, so a
    // dependent's pre-wait reads overlap this kernel alone, never an earlier one.
    pdl_launch_dependents();
    if (warp == 0) {
        for (int s = 0; s < nst; ++s) {
            const int j = c0 + s * G;
            if (j < n_heads) issue_inputs(a, maps, L, j, ins + s * L.bytes, &sh.in_full[s], lane);
        }
    }

    // tokens taken per sequence: all T, or the caller's accepted count (read one head ahead)
    auto tokens_of = [&](int j) {
        return a.accepted ? min(max(a.accepted[j / a.H_v], 0), T) : T;
    };
    int tb_next = c0 < n_heads ? tokens_of(c0) : 0;

    bool ok = true;
    int tok = 0;  // tokens processed by this CTA: parity selects the partial-sum buffer
    int k = 0;
#pragma unroll 1
    for (int j = c0; j < n_heads; j += G, ++k) {
        const int is = k % nst, hp = k & 1;
        const int b = j / a.H_v, h = j % a.H_v;
        const int Tb = tb_next;  // tokens of this head
        if (j + G < n_heads) tb_next = tokens_of(j + G);
        char *in = ins + is * L.bytes;
        // Several tokens per head: the previous head's readers of the per-token
        // rows are done before they are overwritten.  One token: slots alternate.
        if (T > 1) __syncthreads();
        ok &= mbar_wait_bounded(&sh.in_full[is], static_cast<uint32_t>(k / nst) & 1u);

        // A. for every token: conv + SiLU and L2-norm partial sums (q/k threads);
        //    decay, v and the output gate w * silu(z) (other threads)
        {
            const float *win = reinterpret_cast<const float *>(in + L.win);
            const float4 *cwv = reinterpret_cast<const float4 *>(in + L.cw);
            // softplus gates: A = exp(A_log); lower-bound gate: A = the scale a
            const float A_raw = reinterpret_cast<const float *>(in + L.alog)[h & 3];
            const float A = a.lb_gate ? A_raw : __expf(A_raw);
            const int seg = qk_thr ? 0 : 2;  // q (and k) or v channels
            float w0[KM1], w1[KM1];
#pragma unroll
            for (int r = 0; r < KM1; ++r) {
                w0[r] = win[(r * 3 + seg) * SD + ch];
                w1[r] = qk_thr ? win[(r * 3 + 1) * SD + ch] : 0.0f;
            }
            const float4 cw0 = cwv[seg * SD + ch];
            const float4 cw1 = qk_thr ? cwv[SD + ch] : make_float4(0.f, 0.f, 0.f, 0.f);
            // dt_bias of this thread's gate: per channel (softplus KDA), per head (GDN), or the
            // lower bound (per head) of the bounded gate
            const float dt = dt_per_channel(a) ? (qk_thr ? 0.0f : reinterpret_cast<const float *>(in + L.dt)[ch])
                                               : reinterpret_cast<const float *>(in + L.dt)[h & 3];
#pragma unroll 1
            for (int t = 0; t < Tb; ++t) {
                const int sl = T > 1 ? t : hp;
                const char *qkv = in + L.qkv + t * 3 * SD * es;
                if (qk_thr) {
                    const float xq = smem_in(qkv, ch, a.in_bf16);
                    const float xk = smem_in(qkv, SD + ch, a.in_bf16);
                    const float q = conv4_silu_fast(cw0, w0, xq);
                    const float kk = conv4_silu_fast(cw1, w1, xk);
                    w0[0] = w0[1]; w0[1] = w0[2]; w0[2] = xq;
                    w1[0] = w1[1]; w1[1] = w1[2]; w1[2] = xk;
                    sh.q[sl][ch] = q;
                    sh.k[sl][ch] = kk;
                    float sq = q * q, sk = kk * kk, sqk = q * kk;
                    if (tid == 0) {
                        if (!a.kda)
                            sh.a[sl][0] = __expf(-A * softplus_fast(smem_in(in + L.f + t * 16, h & (per16 - 1),
                                                                       a.in_bf16) + dt));
                        sh.beta[sl] = sigmoid_fast(smem_in(in + L.beta + t * 16, h & (per16 - 1), a.in_bf16));
                    }
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) {
                        sq += __shfl_xor_sync(0xffffffffu, sq, off);
                        sk += __shfl_xor_sync(0xffffffffu, sk, off);
                        sqk += __shfl_xor_sync(0xffffffffu, sqk, off);
                    }
                    if (lane == 0) {
                        sh.red3[sl][warp][0] = sq;
                        sh.red3[sl][warp][1] = sk;
                        sh.red3[sl][warp][2] = sqk;
                    }
                } else {
                    if (a.kda) {
                        const float fv = smem_in(in + L.f + t * SD * es, ch, a.in_bf16);
                        sh.a[sl][ch] = a.lb_gate ? __expf(dt * sigmoid_fast(-A * fv)) : __expf(-A * softplus_fast(fv + dt));
                    }
                    const float xv = smem_in(qkv, 2 * SD + ch, a.in_bf16);
                    sh.v[sl][ch] = conv4_silu_fast(cw0, w0, xv);
                    w0[0] = w0[1]; w0[1] = w0[2]; w0[2] = xv;
                    const float zv = smem_in(in + L.z + t * SD * es, ch, a.in_bf16);
                    sh.gz[sl][ch] = nw * (a.sig_gate ? sigmoid_fast(zv) : silu_fast(zv));
                }
                if (a.conv_hist) {  // the window after token t
                    float *chh = a.conv_hist + (static_cast<size_t>(t) * a.B + b) * KM1 * C;
#pragma unroll
                    for (int r = 0; r < KM1; ++r) {
                        chh[static_cast<size_t>(r) * C + seg * a.H_qk * SD + h * SD + ch] = w0[r];
                        if (qk_thr) chh[static_cast<size_t>(r) * C + a.H_qk * SD + h * SD + ch] = w1[r];
                    }
                }
            }
            if (a.conv_out && Tb > 0) {  // the window after the last token
                float *co = a.conv_out + static_cast<size_t>(b) * KM1 * C;
#pragma unroll
                for (int r = 0; r < KM1; ++r) {
                    co[static_cast<size_t>(r) * C + seg * a.H_qk * SD + h * SD + ch] = w0[r];
                    if (qk_thr) co[static_cast<size_t>(r) * C + a.H_qk * SD + h * SD + ch] = w1[r];
                }
            }
        }

        // the state tile (its copy overlapped phase A)
        ok &= mbar_wait_bounded(&sh.tile_full, static_cast<uint32_t>(k) & 1u);
        float4 st[ROWS];
#pragma unroll
        for (int r = 0; r < ROWS; ++r) st[r] = *reinterpret_cast<const float4 *>(tile + (row0 + r) * SD + col0);
        __syncthreads();

        // The tile is in registers everywhere: bring in the CTA's next head.
        if (tid == 0 && j + G < n_heads) {
            fence_proxy_async_smem();
            mbar_expect_tx(&sh.tile_full, TILE_BYTES);
            tma_load_1d(tile, a.state_in + static_cast<size_t>(j + G) * SD * SD, TILE_BYTES, &sh.tile_full);
        }
        // The head's input stage is read out: refill it nst heads ahead.
        if (warp == 0) {
            const int jr = j + nst * G;
            if (jr < n_heads) {
                if (lane == 0) fence_proxy_async_smem();
                __syncwarp();
                issue_inputs(a, maps, L, jr, in, &sh.in_full[is], lane);
            }
        }

#pragma unroll 1
        for (int t = 0; t < Tb; ++t, ++tok) {
            const int sl = T > 1 ? t : hp;
            float *red_k = red + (n_red(T) > 1 ? (tok & 1) : 0) * 2 * CW * SD;
            float *red_q = red_k + CW * SD;
            const size_t e = (static_cast<size_t>(b) * T + t) * a.H_v + h;  // (b, t, h)

            float Sq = 0.f, Sk = 0.f, Sqk = 0.f;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                Sq += sh.red3[sl][w][0];
                Sk += sh.red3[sl][w][1];
                Sqk += sh.red3[sl][w][2];
            }
            const float rq = a.q_scale * rsqrtf(Sq + a.eps_l2);
            const float rk = rsqrtf(Sk + a.eps_l2);
            const float kq = Sqk * rq * rk;

            // B. decay and the two column reductions over this warp's 16 rows
            float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
            for (int r4 = 0; r4 < ROWS / 4; ++r4) {
                const float4 k4 = *reinterpret_cast<const float4 *>(&sh.k[sl][row0 + 4 * r4]);
                const float4 q4 = *reinterpret_cast<const float4 *>(&sh.q[sl][row0 + 4 * r4]);
                const float a0 = sh.a[sl][0];
                float4 a4 = make_float4(a0, a0, a0, a0);
                if (a.kda) a4 = *reinterpret_cast<const float4 *>(&sh.a[sl][row0 + 4 * r4]);
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
            *reinterpret_cast<float4 *>(red_k + warp * SD + col0) = pk;
            *reinterpret_cast<float4 *>(red_q + warp * SD + col0) = pq;
            __syncthreads();

            // Column sums of this lane's four columns (every warp), u = beta (v - St^T k),
            // o = St^T q + (k.q) u, and the sum of o^2 over the head's 128 columns.
            const float beta = sh.beta[sl];
            float4 u4 = *reinterpret_cast<const float4 *>(&sh.v[sl][col0]);
#pragma unroll
            for (int w = 0; w < CW; ++w) {
                const float4 ak = *reinterpret_cast<const float4 *>(red_k + w * SD + col0);
                u4.x -= ak.x; u4.y -= ak.y; u4.z -= ak.z; u4.w -= ak.w;
            }
            u4.x *= beta; u4.y *= beta; u4.z *= beta; u4.w *= beta;
            float4 o4 = make_float4(kq * u4.x, kq * u4.y, kq * u4.z, kq * u4.w);
#pragma unroll
            for (int w = 0; w < CW; ++w) {
                const float4 aq = *reinterpret_cast<const float4 *>(red_q + w * SD + col0);
                o4.x += aq.x; o4.y += aq.y; o4.z += aq.z; o4.w += aq.w;
            }
            float p = o4.x * o4.x + o4.y * o4.y + o4.z * o4.z + o4.w * o4.w;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);

            // gated RMSNorm output, written by one warp per token
            if (a.out && warp == (t & (CW - 1))) {
                const float rinv = rsqrtf(p * (1.0f / SD) + a.eps_norm);
                const float4 g4 = *reinterpret_cast<const float4 *>(&sh.gz[sl][col0]);
                store_out4(a.out, e * SD + col0, a.out_bf16, o4.x * rinv * g4.x, o4.y * rinv * g4.y,
                           o4.z * rinv * g4.z, o4.w * rinv * g4.w);
            }

            // state update and stores
#pragma unroll
            for (int r4 = 0; r4 < ROWS / 4; ++r4) {
                const float4 k4 = *reinterpret_cast<const float4 *>(&sh.k[sl][row0 + 4 * r4]);
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
            else if (a.state_out && t == Tb - 1)
                dst = a.state_out + static_cast<size_t>(j) * SD * SD;
            if (dst) {
#pragma unroll
                for (int r = 0; r < ROWS; ++r)
                    __stcs(reinterpret_cast<float4 *>(dst + (row0 + r) * SD + col0), st[r]);
            }
        }
    }
    if (!ok && lane == 0) atomicOr(&g_stream_error, 1u);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int smem_bytes(int T, int es, int kda, int nst)
{
    return 128 + SH_BYTES + static_cast<int>(TILE_BYTES) + nst * in_layout(T, es, kda, kda).bytes +
           n_red(T) * 2 * CW * SD * 4;
}

// Two input stages when two CTAs per SM still fit, else one.
int stages_for(int T, int es, int kda)
{
    return smem_bytes(T, es, kda, 2) <= (SMEM_PER_SM - 2 * 1024) / 2 ? 2 : 1;
}

}  // namespace

bool stream_eligible(const StepArgs &a)
{
    const size_t es = a.in_bf16 ? 2 : 4;
    // per-head scalars travel as 16-byte rows: the row pitch must be a multiple of 16 bytes
    const bool rows16 = (static_cast<size_t>(a.H_v) * es) % 16 == 0 && a.H_v % 4 == 0;
    bool ok = aligned16(a.qkv) && (static_cast<size_t>(a.C) * es) % 16 == 0 && aligned16(a.z) &&
              aligned16(a.conv_in) && aligned16(a.conv_w) && aligned16(a.beta) && aligned16(a.f) &&
              aligned16(a.dt_bias) && aligned16(a.A_log) && rows16 && a.H_qk == a.H_v;
    return ok && a.T >= 1 && a.T <= MAX_T && a.Ts == a.T && static_cast<long long>(a.B) * a.T * KM1 < (1LL << 31);
}

bool plan_stream(int D, int B, int H_v, int group, int num_sms, StepPlan *plan)
{
    const long units = static_cast<long>(B) * H_v;
    // From 65 units the state staged by TMA beats the register-resident slab and
    // warp-column kernels on the 34-layer chain (us a launch, L2 flushed per step;
    // B3 H32: 5.55 against 9.29, B4: 5.61 against 9.53, B8: 8.93 against 18.75); at
    // 64 units (B2 H32) the two-slab kernel stays ahead, 5.17 against 5.37.
    (void)num_sms;
    if (D != SD || group != 1 || units <= 64 || units >= (1L << 24)) return false;
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
    if (a.gate_lr) return cudaErrorInvalidValue;  // in-kernel gates: slab kernel only
    const int es = a.in_bf16 ? 2 : 4;
    const CUtensorMapDataType ty = a.in_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const uint64_t H = static_cast<uint64_t>(a.H_v), BT = static_cast<uint64_t>(a.B) * a.T;
    const uint32_t T = static_cast<uint32_t>(a.T), per16 = 16 / es;
    InMaps m;
    bool ok = true;
    {   // q, k, v rows: {channel within segment, segment, row b*T+t}
        const uint64_t dim[3] = {H * SD, 3, BT};
        const uint64_t str[2] = {H * SD * es, static_cast<uint64_t>(a.C) * es};
        const uint32_t box[3] = {SD, 3, T};
        ok = ok && encode_tiled(&m.qkv, ty, 3, a.qkv, dim, str, box);
    }
    {   // conv window: {channel within segment, segment, row b*3+r}
        const uint64_t dim[3] = {H * SD, 3, static_cast<uint64_t>(a.B) * KM1};
        const uint64_t str[2] = {H * SD * 4, static_cast<uint64_t>(a.C) * 4};
        const uint32_t box[3] = {SD, 3, KM1};
        ok = ok && encode_tiled(&m.win, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.conv_in, dim, str, box);
    }
    {   // rows of SD per (token, head): z, and the gate rows when per channel
        const uint64_t dim[3] = {SD, H, BT};
        const uint64_t str[2] = {SD * static_cast<uint64_t>(es), H * SD * es};
        const uint32_t box[3] = {SD, 1, T};
        ok = ok && encode_tiled(&m.z, ty, 3, a.z, dim, str, box);
        if (a.kda) ok = ok && encode_tiled(&m.f, ty, 3, a.f, dim, str, box);
    }
    {   // one scalar per (token, head): beta, and the gate when per head
        const uint64_t dim[2] = {H, BT};
        const uint64_t str[1] = {H * es};
        const uint32_t box[2] = {per16, T};
        ok = ok && encode_tiled(&m.beta, ty, 2, a.beta, dim, str, box);
        if (!a.kda) ok = ok && encode_tiled(&m.f, ty, 2, a.f, dim, str, box);
    }
    if (!ok) return cudaErrorInvalidValue;

    static bool attr_set[64];  // per device; benign race: every writer sets the same value
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem_bytes(MAX_T, 4, 1, MAX_STAGES));
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const int n_heads = a.B * a.H_v;
    const int nst = stages_for(a.T, es, a.kda);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid < n_heads ? plan.grid : n_heads, 1, 1);
    cfg.blockDim = dim3(NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = smem_bytes(a.T, es, a.kda, nst);
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
    return cudaLaunchKernelEx(&cfg, stream_kernel, a, m, n_heads, nst);
}

unsigned int take_stream_error()
{
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_stream_error, sizeof(v)) != cudaSuccess) return ~0u;
    if (v && cudaMemcpyToSymbol(g_stream_error, &zero, sizeof(zero)) != cudaSuccess) return ~0u;
    return v;
}

}  // namespace gdn
