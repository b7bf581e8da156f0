// Recurrent KDA / Gated DeltaNet step on sm_103a, column-slab form: decode
// (T = 1), verify (T <= 4, per-token states) and in-place multi-token runs.
// Used when there are too few (sequence, head) units to fill the GPU with
// whole heads (single-sequence decode) and for grouped heads.
//
// One CTA owns a column slab of W value columns of one (sequence, value head)
// state [D, D] (fp32, row = key channel).  The delta rule reduces over key
// rows inside a column ("llama.cpp PR #84": one state column per warp in the
// recurrent kernel), so a CTA that holds every key row of its columns needs no
// other CTA for the update; only the gated RMSNorm needs the whole head, and
// the D / W slabs of a head exchange one partial sum of squares through
// distributed shared memory inside a thread-block cluster.
//
// Per CTA:
//   before the dependency wait (programmatic dependent launch): the state slab
//   (128-bit loads into registers), the conv windows, conv weights and gate
//   parameters -- nothing a preceding kernel on the stream writes;
//   after it, per token, with the next token's inputs already in flight:
//   1. conv window (K = 4) + SiLU for the head's q and k channels and the
//      slab's v channels, L2-norm partial sums, per-channel or per-head decay,
//      beta;
//   2. St = Diag(alpha) S in registers with both column reductions St^T k and
//      St^T q in one pass (warp shuffles, then one shared-memory round);
//   3. u = beta (v - St^T k); o = St^T q + (k.q) u  (= S_new^T q);
//   4. S_new = St + k u^T stored with 128-bit streaming stores, which do not
//      wait for the norm;
//   5. gated RMSNorm over the head's D columns (one partial sum per slab,
//      exchanged inside the cluster).
// The final conv window is written right after the last token's conv, behind a
// cluster barrier that every CTA passes once its window reads are done.  The
// state stays in registers across the T tokens of a verify, so verify and T
// decode calls run the same arithmetic per token.
#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

using namespace dev;

constexpr int KM1 = 3;  // conv window rows kept between calls (conv_K - 1)

__device__ unsigned int g_step_error;  // bit 0: a bounded mbarrier wait gave up

// Asks L2 to fetch every 128-byte line holding a byte of [p, p + bytes), the lanes
// of a warp taking alternate lines.  Nothing comes back to the thread, so this may
// run before the dependency wait on rows the previous kernel is still writing: L2 is
// the point of coherence, and the loads after the wait read the lines as written.
// 8 bf16 weights (16 bytes of shared memory) times 8 fp32 values (shared memory)
__device__ __forceinline__ float dot8_bf16(const unsigned char *w16, const float *x8)
{
    const uint4 w = *reinterpret_cast<const uint4 *>(w16);
    const float4 xa = *reinterpret_cast<const float4 *>(x8);
    const float4 xb = *reinterpret_cast<const float4 *>(x8 + 4);
    const float2 w0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w.x));
    const float2 w1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w.y));
    const float2 w2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w.z));
    const float2 w3 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w.w));
    float acc = w0.x * xa.x;
    acc = fmaf(w0.y, xa.y, acc);
    acc = fmaf(w1.x, xa.z, acc);
    acc = fmaf(w1.y, xa.w, acc);
    acc = fmaf(w2.x, xb.x, acc);
    acc = fmaf(w2.y, xb.y, acc);
    acc = fmaf(w3.x, xb.z, acc);
    return fmaf(w3.y, xb.w, acc);
}

__device__ __forceinline__ void prefetch_l2_lines(const void *p, size_t bytes, int lane)
{
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(p) & ~static_cast<uintptr_t>(127);
    const uintptr_t a1 = reinterpret_cast<uintptr_t>(p) + bytes;
    for (uintptr_t ad = a0 + 128u * static_cast<uintptr_t>(lane); ad < a1; ad += 32u * 128u)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(ad));
}


template <int CQ, int CV>
struct TokenIn {
    float xq[CQ], xk[CQ], fq[CQ], xv[CV];
    float z[4];
    float beta, fh;
};

// GATES: the low-rank gates computed in the kernel (StepArgs::gate_lr), a separate
// instantiation so the plain step keeps its own code.
template <int D, int W, int NT, bool GATES>
__global__ void __launch_bounds__(NT, (256 / NT) > 0 ? (256 / NT) : 1) step_kernel(const StepArgs a)
{
    constexpr int TPR = W / 4;          // threads per state row, one float4 each
    constexpr int RG = NT / TPR;        // row groups
    constexpr int R = D / RG;           // rows per thread
    constexpr int NWARP = NT / 32;
    constexpr int NSLAB = D / W;
    constexpr int CQ = (D + NT - 1) / NT;  // q/k channel pairs per thread
    constexpr int CV = (W + NT - 1) / NT;  // v channels per thread
    static_assert(W % 4 == 0 && 32 % TPR == 0 && NT % 32 == 0 && RG * R == D, "tiling");

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cg = tid % TPR, rg = tid / TPR;
    const int slab = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int hq = h / a.group;
    const bool clustered = NSLAB * a.group > 1;
    const bool qk_owner = (slab == 0) && (h % a.group == 0);  // writes shared q/k conv rows
    const int C = a.C;
    const int tv = (tid + NT - (D % NT)) % NT;  // spreads v channels over idle threads

    __shared__ float q_s[D], k_s[D], a_s[D], v_s[W];
    __shared__ float red3[NWARP][3];
    __shared__ __align__(16) float red_k[NWARP][W];
    __shared__ __align__(16) float red_q[NWARP][W];
    __shared__ float rms_slot[2][NSLAB];
    __shared__ __align__(8) uint64_t rms_bar[2];  // completed by the slabs' pushes of token parity
    __shared__ float beta_s;
    __shared__ float z_s[GATES ? W : 1];
    __shared__ float f_s[GATES ? D : 1];     // in-kernel gates: the head's f
    __shared__ __align__(8) uint64_t f_bar;  // completed by the slabs' pushes of their f share
    // in-kernel gates (a.gate_lr): the W_fb rows of the slab's W key channels, the W_gb
    // rows of its W value columns (each 2R + 16 bytes), then the lr row of the sequence
    extern __shared__ __align__(16) unsigned char gsm[];

    uint32_t rank0 = 0;  // cluster rank of slab 0 of this head
    if (clustered) {
        rank0 = cluster_rank() - slab;
        if (tid == 0) {
            mbar_init(&rms_bar[0], 1);
            mbar_init(&rms_bar[1], 1);
            if (GATES) mbar_init(&f_bar, 1);
            fence_mbar_init();
        }
    }

    bool ok = true;  // false once a bounded wait gave up

    // ---- before the dependency wait: state slab, conv windows, parameters
    const size_t head = static_cast<size_t>(b) * a.H_v + h;
    const size_t col0 = static_cast<size_t>(slab) * W + 4 * cg;
    float4 st[R];
    {
        const float *S = a.state_in + head * D * D + col0;
#pragma unroll
        for (int r = 0; r < R; ++r)
            st[r] = __ldcs(reinterpret_cast<const float4 *>(S + static_cast<size_t>(rg + RG * r) * D));
    }
    float wq[CQ][KM1], wk[CQ][KM1], wv[CV][KM1];
    float4 cwq[CQ], cwk[CQ], cwv[CV];
    float dtb[CQ];
    // softplus gates: A = exp(A_log); lower-bound gate: A = the scale a, lbv = the bound
    const float A = a.lb_gate ? a.A_log[h] : __expf(a.A_log[h]);
    const float lbv = a.lb_gate ? a.dt_bias[h] : 0.0f;
#pragma unroll
    for (int m = 0; m < CQ; ++m) {
        const int i = tid + m * NT;
        if (i < D) {
            const int cq = hq * D + i, ck = a.H_qk * D + hq * D + i;
#pragma unroll
            for (int r = 0; r < KM1; ++r) {
                wq[m][r] = a.conv_in[(static_cast<size_t>(b) * KM1 + r) * C + cq];
                wk[m][r] = a.conv_in[(static_cast<size_t>(b) * KM1 + r) * C + ck];
            }
            cwq[m] = reinterpret_cast<const float4 *>(a.conv_w)[cq];
            cwk[m] = reinterpret_cast<const float4 *>(a.conv_w)[ck];
            dtb[m] = a.kda && !a.lb_gate ? a.dt_bias[static_cast<size_t>(h) * D + i] : 0.0f;
        }
    }
#pragma unroll
    for (int m = 0; m < CV; ++m) {
        const int j = tv + m * NT;
        if (j < W) {
            const int cv = 2 * a.H_qk * D + h * D + slab * W + j;
#pragma unroll
            for (int r = 0; r < KM1; ++r)
                wv[m][r] = a.conv_in[(static_cast<size_t>(b) * KM1 + r) * C + cv];
            cwv[m] = reinterpret_cast<const float4 *>(a.conv_w)[cv];
        }
    }
    float nw[4] = {0.f, 0.f, 0.f, 0.f};
    if (rg == 0) {
#pragma unroll
        for (int c = 0; c < 4; ++c) nw[c] = a.norm_w[col0 + c];
    }
    const float dtb_head = a.kda ? 0.0f : a.dt_bias[h];

    // In-kernel gates: the weight rows they need go to shared memory now (read-only).
    constexpr bool gates = GATES;
    const int GR = a.gate_rank, GS = 2 * GR + 16;
    if constexpr (GATES) {
        const int cpr = GR / 8;  // 16-byte pieces a row
        for (int i = tid; i < 2 * W * cpr; i += NT) {
            const int r = i / cpr, c = i - r * cpr;
            const bool fb = r < W;
            const size_t grow = static_cast<size_t>(h) * D + slab * W + (fb ? r : r - W);
            cp_async16(gsm + r * GS + c * 16,
                       static_cast<const __nv_bfloat16 *>(fb ? a.w_fb : a.w_gb) + grow * GR + c * 8);
        }
    }

    // The rows of the first tokens' inputs are asked into L2 now, so that the loads
    // after the wait find them there (a warp per input segment).
    {
        const int ntok = min(a.T, 4);
        const size_t esz = a.in_bf16 ? 2 : 4;
        const char *qkv = static_cast<const char *>(a.qkv);
        for (int s = warp; s < 6 * ntok; s += NWARP) {
            const size_t bt = static_cast<size_t>(b) * a.Ts + s / 6;
            const size_t row = bt * C, bth = bt * a.H_v + h;
            const void *p = nullptr;
            size_t n = 0;
            switch (s % 6) {
            case 0: p = qkv + (row + hq * D) * esz; n = D; break;
            case 1: p = qkv + (row + static_cast<size_t>(a.H_qk + hq) * D) * esz; n = D; break;
            case 2: p = qkv + (row + 2 * static_cast<size_t>(a.H_qk) * D + h * D + slab * W) * esz; n = W; break;
            case 3:
                if (gates) break;
                p = static_cast<const char *>(a.f) + (a.kda ? bth * D : bth) * esz;
                n = a.kda ? D : 1;
                break;
            case 4:
                if (gates) break;
                p = static_cast<const char *>(a.z) + (bth * D + slab * W) * esz;
                n = W;
                break;
            default: p = static_cast<const char *>(a.beta) + bth * esz; n = 1; break;
            }
            prefetch_l2_lines(p, n * esz, lane);
        }
    }

    // Every CTA's reads of the conv window (and its barrier set-up) are ordered before
    // the window's in-place update, which the writing threads make after this barrier's
    // wait.  Within a CTA each window channel is read and written by the same thread.
    if (clustered) cluster_arrive_release();

    // ---- inputs may be written by the previous kernel on the stream
    pdl_wait();
    // Dependents launch only once this grid has passed its own dependency wait, so a
    // dependent's pre-wait reads overlap this kernel alone, never an earlier one.
    pdl_launch_dependents();

    // All inputs of token t in one round of independent loads.
    auto load_token = [&](int t, TokenIn<CQ, CV> &in) {
        const size_t bt = static_cast<size_t>(b) * a.Ts + t;
        const size_t row = bt * C;
        const size_t bth = bt * a.H_v + h;
#pragma unroll
        for (int m = 0; m < CQ; ++m) {
            const int i = tid + m * NT;
            if (i < D) {
                in.xq[m] = ld_in(a.qkv, row + hq * D + i, a.in_bf16);
                in.xk[m] = ld_in(a.qkv, row + a.H_qk * D + hq * D + i, a.in_bf16);
                in.fq[m] = a.kda && !gates ? ld_in(a.f, bth * D + i, a.in_bf16) : 0.0f;
            }
        }
#pragma unroll
        for (int m = 0; m < CV; ++m) {
            const int j = tv + m * NT;
            if (j < W) in.xv[m] = ld_in(a.qkv, row + 2 * a.H_qk * D + h * D + slab * W + j, a.in_bf16);
        }
        if (rg == 0 && !gates) {
#pragma unroll
            for (int c = 0; c < 4; ++c) in.z[c] = ld_in(a.z, bth * D + col0 + c, a.in_bf16);
        }
        if (tid == 0) {
            in.beta = ld_in(a.beta, bth, a.in_bf16);
            in.fh = a.kda ? 0.0f : ld_in(a.f, bth, a.in_bf16);
        }
    };

    TokenIn<CQ, CV> cur;
    // tokens taken for this sequence: all T, or the caller's accepted count
    const int Tb = a.accepted ? min(max(a.accepted[b], 0), a.T) : a.T;
    if (Tb > 0) load_token(0, cur);
    if (clustered) cluster_wait_acquire();  // every CTA's barriers and window reads
    if constexpr (GATES) {
        // The slab's 2W outputs: f of key channels slab W + o (o < W), which every slab
        // of the head needs for its decay, and z of its own value columns (o >= W); NT /
        // (2W) threads an output, 16-byte pieces of the rank taken round robin.
        float *lr_s = reinterpret_cast<float *>(gsm + 2 * W * GS);
        const size_t bth0 = static_cast<size_t>(b) * a.Ts * a.H_v + h;  // token 0
        for (int i = tid; i < 2 * GR; i += NT) lr_s[i] = a.gate_lr[static_cast<size_t>(b) * 2 * GR + i];
        cp_async_wait_all();
        __syncthreads();
        constexpr int PARTS = NT / (2 * W);
        static_assert(PARTS >= 1 && 32 % PARTS == 0, "gate output split");
        const int o = tid / PARTS, part = tid % PARTS;
        const float *x = lr_s + (o < W ? 0 : GR);
        float g0 = 0.f, g1 = 0.f;
        int c = part;
        for (; c + PARTS < GR / 8; c += 2 * PARTS) {
            g0 += dot8_bf16(gsm + o * GS + c * 16, x + c * 8);
            g1 += dot8_bf16(gsm + o * GS + (c + PARTS) * 16, x + (c + PARTS) * 8);
        }
        if (c < GR / 8) g0 += dot8_bf16(gsm + o * GS + c * 16, x + c * 8);
        float gv = g0 + g1;
#pragma unroll
        for (int off = PARTS >> 1; off > 0; off >>= 1) gv += __shfl_xor_sync(0xffffffffu, gv, off);
        if (NSLAB > 1 && tid == 0) mbar_expect_tx(&f_bar, D * 4);
        if (part == 0) {
            if (o < W) {
                const int ch = slab * W + o;
                if (NSLAB > 1) {
                    for (int d = 0; d < NSLAB; ++d) st_async_remote(&f_s[ch], rank0 + d, gv, &f_bar);
                } else {
                    f_s[ch] = gv;
                }
                if (a.gate_f) a.gate_f[bth0 * D + ch] = gv;
            } else {
                z_s[o - W] = gv;
                if (a.gate_z) a.gate_z[bth0 * D + slab * W + (o - W)] = gv;
            }
        }
        __syncthreads();
        if (NSLAB > 1) ok &= mbar_wait_cluster_bounded(&f_bar, 0u);
#pragma unroll
        for (int m = 0; m < CQ; ++m) {
            const int i = tid + m * NT;
            if (i < D) cur.fq[m] = f_s[i];
        }
        if (rg == 0) {
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) cur.z[c4] = z_s[4 * cg + c4];
        }
    }

#pragma unroll 1
    for (int t = 0; t < Tb; ++t) {
        if (t > 0) __syncthreads();  // previous token's shared-memory reads are done
        TokenIn<CQ, CV> nxt;
        if (t + 1 < Tb) load_token(t + 1, nxt);
        const size_t bth = (static_cast<size_t>(b) * a.Ts + t) * a.H_v + h;

        // 1. conv + SiLU, norms' partial sums, gates
        float sq = 0.f, sk = 0.f, sqk = 0.f;
#pragma unroll
        for (int m = 0; m < CQ; ++m) {
            const int i = tid + m * NT;
            if (i < D) {
                const float q = conv4_silu_fast(cwq[m], wq[m], cur.xq[m]);
                const float k = conv4_silu_fast(cwk[m], wk[m], cur.xk[m]);
                wq[m][0] = wq[m][1]; wq[m][1] = wq[m][2]; wq[m][2] = cur.xq[m];
                wk[m][0] = wk[m][1]; wk[m][1] = wk[m][2]; wk[m][2] = cur.xk[m];
                q_s[i] = q;
                k_s[i] = k;
                sq = fmaf(q, q, sq);
                sk = fmaf(k, k, sk);
                sqk = fmaf(q, k, sqk);
                if (a.kda)
                    a_s[i] = a.lb_gate ? __expf(lbv * sigmoid_fast(-A * cur.fq[m]))
                                       : __expf(-A * softplus_fast(cur.fq[m] + dtb[m]));
            }
        }
#pragma unroll
        for (int m = 0; m < CV; ++m) {
            const int j = tv + m * NT;
            if (j < W) {
                v_s[j] = conv4_silu_fast(cwv[m], wv[m], cur.xv[m]);
                wv[m][0] = wv[m][1]; wv[m][1] = wv[m][2]; wv[m][2] = cur.xv[m];
            }
        }
        if (tid == 0) {
            if (!a.kda) a_s[0] = __expf(-A * softplus_fast(cur.fh + dtb_head));
            beta_s = sigmoid_fast(cur.beta);
        }
        // the window after the last token (commit): every reader has passed the barrier above
        if (a.conv_out && t == Tb - 1) {
            float *co = a.conv_out + static_cast<size_t>(b) * KM1 * C;
#pragma unroll
            for (int m = 0; m < CQ; ++m) {
                const int i = tid + m * NT;
                if (i < D && qk_owner) {
                    const int cq = hq * D + i, ck = a.H_qk * D + hq * D + i;
#pragma unroll
                    for (int r = 0; r < KM1; ++r) {
                        co[static_cast<size_t>(r) * C + cq] = wq[m][r];
                        co[static_cast<size_t>(r) * C + ck] = wk[m][r];
                    }
                }
            }
#pragma unroll
            for (int m = 0; m < CV; ++m) {
                const int j = tv + m * NT;
                if (j < W) {
                    const int cv = 2 * a.H_qk * D + h * D + slab * W + j;
#pragma unroll
                    for (int r = 0; r < KM1; ++r) co[static_cast<size_t>(r) * C + cv] = wv[m][r];
                }
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            sq += __shfl_xor_sync(0xffffffffu, sq, off);
            sk += __shfl_xor_sync(0xffffffffu, sk, off);
            sqk += __shfl_xor_sync(0xffffffffu, sqk, off);
        }
        if (lane == 0) {
            red3[warp][0] = sq;
            red3[warp][1] = sk;
            red3[warp][2] = sqk;
        }
        __syncthreads();

        float Sq = 0.f, Sk = 0.f, Sqk = 0.f;
#pragma unroll
        for (int w = 0; w < NWARP; ++w) {
            Sq += red3[w][0];
            Sk += red3[w][1];
            Sqk += red3[w][2];
        }
        const float rq = a.q_scale * rsqrtf(Sq + a.eps_l2);
        const float rk = rsqrtf(Sk + a.eps_l2);
        const float kq = Sqk * rq * rk;
        const float beta = beta_s;

        // 2. decay and the two column reductions in one pass
        float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int row = rg + RG * r;
            const float al = a_s[a.kda ? row : 0];
            const float kr = k_s[row] * rk, qr = q_s[row] * rq;
            st[r].x *= al; st[r].y *= al; st[r].z *= al; st[r].w *= al;
            pk.x = fmaf(st[r].x, kr, pk.x); pk.y = fmaf(st[r].y, kr, pk.y);
            pk.z = fmaf(st[r].z, kr, pk.z); pk.w = fmaf(st[r].w, kr, pk.w);
            pq.x = fmaf(st[r].x, qr, pq.x); pq.y = fmaf(st[r].y, qr, pq.y);
            pq.z = fmaf(st[r].z, qr, pq.z); pq.w = fmaf(st[r].w, qr, pq.w);
        }
#pragma unroll
        for (int off = TPR; off < 32; off <<= 1) {
            pk.x += __shfl_xor_sync(0xffffffffu, pk.x, off);
            pk.y += __shfl_xor_sync(0xffffffffu, pk.y, off);
            pk.z += __shfl_xor_sync(0xffffffffu, pk.z, off);
            pk.w += __shfl_xor_sync(0xffffffffu, pk.w, off);
            pq.x += __shfl_xor_sync(0xffffffffu, pq.x, off);
            pq.y += __shfl_xor_sync(0xffffffffu, pq.y, off);
            pq.z += __shfl_xor_sync(0xffffffffu, pq.z, off);
            pq.w += __shfl_xor_sync(0xffffffffu, pq.w, off);
        }
        if (lane < TPR) {
            *reinterpret_cast<float4 *>(&red_k[warp][4 * cg]) = pk;
            *reinterpret_cast<float4 *>(&red_q[warp][4 * cg]) = pq;
        }
        __syncthreads();

        // 3. u and o for this thread's four columns
        float kS[4] = {0.f, 0.f, 0.f, 0.f}, qS[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int w = 0; w < NWARP; ++w) {
            const float4 ak = *reinterpret_cast<const float4 *>(&red_k[w][4 * cg]);
            const float4 aq = *reinterpret_cast<const float4 *>(&red_q[w][4 * cg]);
            kS[0] += ak.x; kS[1] += ak.y; kS[2] += ak.z; kS[3] += ak.w;
            qS[0] += aq.x; qS[1] += aq.y; qS[2] += aq.z; qS[3] += aq.w;
        }
        float u[4], o[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            u[c] = beta * (v_s[4 * cg + c] - kS[c]);
            o[c] = fmaf(kq, u[c], qS[c]);
        }

        // 4. state update and stores (they do not wait for the RMS exchange)
        const bool last = (t == Tb - 1);
        float *hist = a.state_hist
            ? a.state_hist + ((static_cast<size_t>(t) * a.B + b) * a.H_v + h) * D * D + col0
            : nullptr;
        float *commit = (a.state_out && last) ? a.state_out + head * D * D + col0 : nullptr;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int row = rg + RG * r;
            const float kr = k_s[row] * rk;
            st[r].x = fmaf(kr, u[0], st[r].x);
            st[r].y = fmaf(kr, u[1], st[r].y);
            st[r].z = fmaf(kr, u[2], st[r].z);
            st[r].w = fmaf(kr, u[3], st[r].w);
            const size_t off = static_cast<size_t>(row) * D;
            if (hist) __stcs(reinterpret_cast<float4 *>(hist + off), st[r]);
            if (commit) __stcs(reinterpret_cast<float4 *>(commit + off), st[r]);
        }

        // 5. gated RMSNorm over the head's D columns.  The D / W slabs push their
        //    partial sums of o^2 into every slab's slot for this token parity and
        //    complete 4 bytes each on that slab's mbarrier; a slab can be at most one
        //    token ahead of the slowest (it needs every partial to finish a token).
        float p = 0.f;
        if (warp == 0) {
            // the slab's columns sit on lanes 0..TPR-1 of warp 0
            if (rg == 0) p = o[0] * o[0] + o[1] * o[1] + o[2] * o[2] + o[3] * o[3];
#pragma unroll
            for (int off = TPR >> 1; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
            p = __shfl_sync(0xffffffffu, p, 0);
        }
        float total = p;
        if (clustered) {
            if (warp == 0) {  // lane s pushes to slab s
                if (lane == 0) mbar_expect_tx(&rms_bar[t & 1], NSLAB * 4);
                if (lane < NSLAB) st_async_remote(&rms_slot[t & 1][slab], rank0 + lane, p, &rms_bar[t & 1]);
            }
            if (rg == 0) {
                ok &= mbar_wait_cluster_bounded(&rms_bar[t & 1], static_cast<uint32_t>(t >> 1) & 1u);
                total = 0.f;
#pragma unroll
                for (int s = 0; s < NSLAB; ++s) total += rms_slot[t & 1][s];
            }
        }
        if (rg == 0 && a.out) {
            const float rinv = rsqrtf(total * (1.0f / D) + a.eps_norm);
            float y[4];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                y[c] = o[c] * rinv * nw[c] * (a.sig_gate ? sigmoid_fast(cur.z[c]) : silu_fast(cur.z[c]));
            store_out4(a.out, bth * D + col0, a.out_bf16, y[0], y[1], y[2], y[3]);
        }

        // conv window after this token (verify history)
        if (a.conv_hist) {
            float *ch = a.conv_hist + (static_cast<size_t>(t) * a.B + b) * KM1 * C;
#pragma unroll
            for (int m = 0; m < CQ; ++m) {
                const int i = tid + m * NT;
                if (i < D && qk_owner) {
                    const int cq = hq * D + i, ck = a.H_qk * D + hq * D + i;
#pragma unroll
                    for (int r = 0; r < KM1; ++r) {
                        ch[static_cast<size_t>(r) * C + cq] = wq[m][r];
                        ch[static_cast<size_t>(r) * C + ck] = wk[m][r];
                    }
                }
            }
#pragma unroll
            for (int m = 0; m < CV; ++m) {
                const int j = tv + m * NT;
                if (j < W) {
                    const int cv = 2 * a.H_qk * D + h * D + slab * W + j;
#pragma unroll
                    for (int r = 0; r < KM1; ++r) ch[static_cast<size_t>(r) * C + cv] = wv[m][r];
                }
            }
        }
        cur = nxt;
    }

    if (!ok) atomicOr(&g_step_error, 1u);
}

// ---------------------------------------------------------------- warp-column form (d = 128)
//
// The same step at d = 128 with every reduction of a token inside one warp: a warp
// owns 8 value columns of the head and all 128 key rows (lane l: rows 4l..4l+3, so
// 32 state values a lane), and computes the conv, the norms and the decay of the
// head's q/k channels for its own rows.  The column sums S_t^T k and S_t^T q of its
// 8 columns are a 16-value reduce-scatter over the warp (16 shuffles), after which
// lanes 2c and 2c+1 hold column c's k-sum (lanes 0..15) or q-sum (lanes 16..31).
// Nothing but the RMS norm's sum over the head's 128 columns leaves the warp:
// through shared memory when one CTA holds the head, else by st.async pushes to
// every CTA of the head inside a cluster, as in the slab form above.
// Scalar maps use the hardware exponential, logarithm and reciprocal.

constexpr int WD = 128;   // key and value width of this form
constexpr int WCOL = 8;   // value columns per warp


struct WIn {
    float q[4], k[4], f[4];
    float vz;  // lanes 0..15: v of column (lane/2)%8; lanes 16..31: z of that column
    float beta, fh;
};

template <int NW>
__global__ void __launch_bounds__(NW * 32) wstep_kernel(const StepArgs a)
{
    constexpr int D = WD;
    constexpr int W = WCOL * NW;     // value columns of the CTA
    constexpr int NSLAB = D / W;     // CTAs per head
    constexpr unsigned FULL = 0xffffffffu;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int slab = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int hq = h / a.group;
    const bool clustered = NSLAB * a.group > 1;
    const bool qk_owner = slab == 0 && h % a.group == 0 && warp == 0;  // writes the q/k window
    const int C = a.C;
    const int r0 = 4 * lane;                 // key rows (channels) of this lane
    const int jc = (lane >> 1) & 7;          // the column whose sums this lane holds
    const bool klane = lane < 16;            // k-sum (and v) lanes; the others q-sum (and z)
    const bool vown = klane && (lane & 1) == 0;  // reads and writes column jc's v window
    const int c0 = slab * W + WCOL * warp;   // first value column of the warp

    __shared__ float4 cw_s[2][4][32];        // conv taps of the head's q and k channels, [i][lane]
    __shared__ float rms_slot[2][NSLAB * NW];  // the warps' sums of o^2, by token parity
    __shared__ __align__(8) uint64_t rms_bar[2];

    uint32_t rank0 = 0;  // cluster rank of slab 0 of this head
    if (NSLAB > 1 || clustered) {
        rank0 = cluster_rank() - slab;
        if (NSLAB > 1 && tid == 0) {
            mbar_init(&rms_bar[0], 1);
            mbar_init(&rms_bar[1], 1);
            fence_mbar_init();
        }
    }
    bool ok = true;

    // ---- before the dependency wait: state, conv windows and taps, parameters
    const size_t head = static_cast<size_t>(b) * a.H_v + h;
    float st[4][WCOL];
    {
        const float *S = a.state_in + head * D * D + c0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 lo = *reinterpret_cast<const float4 *>(S + static_cast<size_t>(r0 + i) * D);
            const float4 hi = *reinterpret_cast<const float4 *>(S + static_cast<size_t>(r0 + i) * D + 4);
            st[i][0] = lo.x; st[i][1] = lo.y; st[i][2] = lo.z; st[i][3] = lo.w;
            st[i][4] = hi.x; st[i][5] = hi.y; st[i][6] = hi.z; st[i][7] = hi.w;
        }
    }
    const int cq = hq * D + r0, ck = (a.H_qk + hq) * D + r0;
    const int cv = 2 * a.H_qk * D + h * D + c0 + jc;
    float wq[4][KM1], wk[4][KM1], wv[KM1] = {0.f, 0.f, 0.f};
#pragma unroll
    for (int r = 0; r < KM1; ++r) {
        const float *row = a.conv_in + (static_cast<size_t>(b) * KM1 + r) * C;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            wq[i][r] = row[cq + i];
            wk[i][r] = row[ck + i];
        }
        if (vown) wv[r] = row[cv];
    }
    for (int e = tid; e < 2 * 4 * 32; e += NW * 32) {
        const int s = e >> 7, i = (e >> 5) & 3, l = e & 31;
        cw_s[s][i][l] = reinterpret_cast<const float4 *>(a.conv_w)[(s ? a.H_qk + hq : hq) * D + 4 * l + i];
    }
    const float4 cwv = vown ? reinterpret_cast<const float4 *>(a.conv_w)[cv] : make_float4(0.f, 0.f, 0.f, 0.f);
    // softplus gates: A = exp(A_log); lower-bound gate: A = the scale a, lbv = the bound
    const float A = a.lb_gate ? a.A_log[h] : __expf(a.A_log[h]);
    const float lbv = a.lb_gate ? a.dt_bias[h] : 0.0f;
    float dtb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) dtb[i] = a.kda && !a.lb_gate ? a.dt_bias[static_cast<size_t>(h) * D + r0 + i] : 0.0f;
    const float dtb_head = a.kda ? 0.0f : a.dt_bias[h];
    const float nw = klane ? 0.0f : a.norm_w[c0 + jc];

    // The first tokens' input rows are asked into L2 before the wait (a warp per segment).
    {
        const int ntok = min(a.T, 4);
        const size_t esz = a.in_bf16 ? 2 : 4;
        const char *qkv = static_cast<const char *>(a.qkv);
        for (int s = warp; s < 6 * ntok; s += NW) {
            const size_t bt = static_cast<size_t>(b) * a.Ts + s / 6;
            const size_t row = bt * C, bth = bt * a.H_v + h;
            const void *p = nullptr;
            size_t n = 0;
            switch (s % 6) {
            case 0: p = qkv + (row + hq * D) * esz; n = D; break;
            case 1: p = qkv + (row + static_cast<size_t>(a.H_qk + hq) * D) * esz; n = D; break;
            case 2: p = qkv + (row + 2 * static_cast<size_t>(a.H_qk) * D + h * D + slab * W) * esz; n = W; break;
            case 3:
                p = static_cast<const char *>(a.f) + (a.kda ? bth * D : bth) * esz;
                n = a.kda ? D : 1;
                break;
            case 4: p = static_cast<const char *>(a.z) + (bth * D + slab * W) * esz; n = W; break;
            default: p = static_cast<const char *>(a.beta) + bth * esz; n = 1; break;
            }
            prefetch_l2_lines(p, n * esz, lane);
        }
    }
    // Every read of the conv window (and the barrier set-up) is ordered before the
    // window's in-place update by the writing warp, which passes this barrier's wait
    // before its first token.
    if (NSLAB > 1 || clustered) cluster_arrive_release();
    __syncthreads();  // conv taps in shared memory; the CTA's own window reads

    // ---- inputs may be written by the previous kernel on the stream
    pdl_wait();
    // Dependents launch only once this grid has passed its own dependency wait, so a
    // dependent's pre-wait reads overlap this kernel alone, never an earlier one.
    pdl_launch_dependents();

    auto load_token = [&](int t, WIn &in) {
        const size_t bt = static_cast<size_t>(b) * a.Ts + t;
        const size_t row = bt * C, bth = bt * a.H_v + h;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            in.q[i] = ld_in(a.qkv, row + cq + i, a.in_bf16);
            in.k[i] = ld_in(a.qkv, row + ck + i, a.in_bf16);
            in.f[i] = a.kda ? ld_in(a.f, bth * D + r0 + i, a.in_bf16) : 0.0f;
        }
        in.vz = klane ? ld_in(a.qkv, row + cv, a.in_bf16) : ld_in(a.z, bth * D + c0 + jc, a.in_bf16);
        in.beta = ld_in(a.beta, bth, a.in_bf16);
        in.fh = a.kda ? 0.0f : ld_in(a.f, bth, a.in_bf16);
    };

    WIn cur;
    const int Tb = a.accepted ? min(max(a.accepted[b], 0), a.T) : a.T;
    if (Tb > 0) load_token(0, cur);
    if (NSLAB > 1 || clustered) cluster_wait_acquire();  // every CTA's barriers and window reads

#pragma unroll 1
    for (int t = 0; t < Tb; ++t) {
        WIn nxt;
        if (t + 1 < Tb) load_token(t + 1, nxt);
        const size_t bth = (static_cast<size_t>(b) * a.Ts + t) * a.H_v + h;

        // 1. conv + SiLU of the lane's q/k channels, their decay, v of column jc, beta
        float q[4], k[4], al[4];
        float sq = 0.f, sk = 0.f, sqk = 0.f;
        const float alh = a.kda ? 0.0f : __expf(-A * softplus_fast(cur.fh + dtb_head));
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 tq = cw_s[0][i][lane], tk = cw_s[1][i][lane];
            float xq = tq.x * wq[i][0];
            xq = fmaf(tq.y, wq[i][1], xq);
            xq = fmaf(tq.z, wq[i][2], xq);
            xq = fmaf(tq.w, cur.q[i], xq);
            float xk = tk.x * wk[i][0];
            xk = fmaf(tk.y, wk[i][1], xk);
            xk = fmaf(tk.z, wk[i][2], xk);
            xk = fmaf(tk.w, cur.k[i], xk);
            q[i] = silu_fast(xq);
            k[i] = silu_fast(xk);
            wq[i][0] = wq[i][1]; wq[i][1] = wq[i][2]; wq[i][2] = cur.q[i];
            wk[i][0] = wk[i][1]; wk[i][1] = wk[i][2]; wk[i][2] = cur.k[i];
            sq = fmaf(q[i], q[i], sq);
            sk = fmaf(k[i], k[i], sk);
            sqk = fmaf(q[i], k[i], sqk);
            al[i] = !a.kda ? alh
                  : a.lb_gate ? __expf(lbv * sigmoid_fast(-A * cur.f[i]))
                              : __expf(-A * softplus_fast(cur.f[i] + dtb[i]));
        }
        float vv = 0.f;
        if (vown) {
            float x = cwv.x * wv[0];
            x = fmaf(cwv.y, wv[1], x);
            x = fmaf(cwv.z, wv[2], x);
            x = fmaf(cwv.w, cur.vz, x);
            vv = silu_fast(x);
            wv[0] = wv[1]; wv[1] = wv[2]; wv[2] = cur.vz;
        }
        vv = __shfl_sync(FULL, vv, lane & ~1);
        const float beta = sigmoid_fast(cur.beta);
        const bool last = (t == Tb - 1);
        // the window after the last token (commit): every reader has passed the barrier above
        if (last && a.conv_out) {
            float *co = a.conv_out + static_cast<size_t>(b) * KM1 * C;
#pragma unroll
            for (int r = 0; r < KM1; ++r) {
                if (qk_owner) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        co[static_cast<size_t>(r) * C + cq + i] = wq[i][r];
                        co[static_cast<size_t>(r) * C + ck + i] = wk[i][r];
                    }
                }
                if (vown) co[static_cast<size_t>(r) * C + cv] = wv[r];
            }
        }

        // 2. decay, and the lane's parts of S_t^T k and S_t^T q (raw q, k; scaled below)
        float red[2 * WCOL];
#pragma unroll
        for (int c = 0; c < 2 * WCOL; ++c) red[c] = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int c = 0; c < WCOL; ++c) {
                st[i][c] *= al[i];
                red[c] = fmaf(st[i][c], k[i], red[c]);
                red[WCOL + c] = fmaf(st[i][c], q[i], red[WCOL + c]);
            }
        }
        // the norms' sums over the head's 128 channels (all lanes)
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            sq += __shfl_xor_sync(FULL, sq, off);
            sk += __shfl_xor_sync(FULL, sk, off);
            sqk += __shfl_xor_sync(FULL, sqk, off);
        }
        // reduce-scatter: after the rounds lane l holds value (l >> 1) summed over the warp
#pragma unroll
        for (int n = WCOL; n >= 1; n >>= 1) {
            const int off = 2 * n;  // 16, 8, 4, 2
            const bool up = (lane & off) != 0;
#pragma unroll
            for (int i = 0; i < n; ++i) {
                const float send = up ? red[i] : red[i + n];
                const float keep = up ? red[i + n] : red[i];
                red[i] = keep + __shfl_xor_sync(FULL, send, off);
            }
        }
        const float tot = red[0] + __shfl_xor_sync(FULL, red[0], 1);
        const float rq = a.q_scale * rsqrtf(sq + a.eps_l2);
        const float rk = rsqrtf(sk + a.eps_l2);
        const float kq = sqk * rq * rk;

        // 3. u (k lanes) and o (q lanes) of column jc
        const float u = beta * (vv - rk * tot);
        const float o = fmaf(kq, __shfl_xor_sync(FULL, u, 16), rq * tot);

        // 4. state update, stores (they do not wait for the RMS exchange)
        float *hist = a.state_hist
            ? a.state_hist + ((static_cast<size_t>(t) * a.B + b) * a.H_v + h) * D * D + c0
            : nullptr;
        float *commit = (a.state_out && last) ? a.state_out + head * D * D + c0 : nullptr;
        float ub[WCOL];
#pragma unroll
        for (int c = 0; c < WCOL; ++c) ub[c] = __shfl_sync(FULL, u, 2 * c);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float kn = k[i] * rk;
#pragma unroll
            for (int c = 0; c < WCOL; ++c) st[i][c] = fmaf(kn, ub[c], st[i][c]);
            const size_t off = static_cast<size_t>(r0 + i) * D;
            const float4 lo = make_float4(st[i][0], st[i][1], st[i][2], st[i][3]);
            const float4 hi = make_float4(st[i][4], st[i][5], st[i][6], st[i][7]);
            if (hist) {
                __stcs(reinterpret_cast<float4 *>(hist + off), lo);
                __stcs(reinterpret_cast<float4 *>(hist + off + 4), hi);
            }
            if (commit) {
                __stcs(reinterpret_cast<float4 *>(commit + off), lo);
                __stcs(reinterpret_cast<float4 *>(commit + off + 4), hi);
            }
        }

        // 5. gated RMSNorm over the head's 128 columns
        float p = (!klane && (lane & 1) == 0) ? o * o : 0.f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(FULL, p, off);
        float total = 0.f;
        const int par = t & 1;
        if (NSLAB == 1) {
            if (lane == 0) rms_slot[par][warp] = p;
            __syncthreads();
        } else {
            // each warp's sum to its slot in every CTA of the head
            if (tid == 0) mbar_expect_tx(&rms_bar[par], NSLAB * NW * 4);
            if (lane < NSLAB)
                st_async_remote(&rms_slot[par][slab * NW + warp], rank0 + lane, p, &rms_bar[par]);
            ok &= mbar_wait_cluster_bounded(&rms_bar[par], static_cast<uint32_t>(t >> 1) & 1u);
        }
#pragma unroll
        for (int s = 0; s < NSLAB * NW; ++s) total += rms_slot[par][s];
        if (!klane && (lane & 1) == 0 && a.out) {
            const float rinv = rsqrtf(total * (1.0f / D) + a.eps_norm);
            const float g = a.sig_gate ? sigmoid_fast(cur.vz) : silu_fast(cur.vz);
            const float y = o * rinv * nw * g;
            const size_t idx = bth * D + c0 + jc;
            if (a.out_bf16)
                reinterpret_cast<__nv_bfloat16 *>(a.out)[idx] = __float2bfloat16_rn(y);
            else
                reinterpret_cast<float *>(a.out)[idx] = y;
        }

        // conv window after this token (verify history)
        if (a.conv_hist) {
            float *ch = a.conv_hist + (static_cast<size_t>(t) * a.B + b) * KM1 * C;
#pragma unroll
            for (int r = 0; r < KM1; ++r) {
                if (qk_owner) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        ch[static_cast<size_t>(r) * C + cq + i] = wq[i][r];
                        ch[static_cast<size_t>(r) * C + ck + i] = wk[i][r];
                    }
                }
                if (vown) ch[static_cast<size_t>(r) * C + cv] = wv[r];
            }
        }
        cur = nxt;
    }

    if (!ok) atomicOr(&g_step_error, 1u);
}

struct Variant {
    int D, W, NT;
    void (*fn)(StepArgs);
    void (*fn_gates)(StepArgs);  // with the in-kernel low-rank gates
    const char *name;
};

#define GDN_VARIANT(D, W, NT) \
    {D, W, NT, step_kernel<D, W, NT, false>, step_kernel<D, W, NT, true>, "step<" #D "," #W ">"}
const Variant kVariants[] = {
    GDN_VARIANT(128, 128, 256), GDN_VARIANT(128, 64, 256), GDN_VARIANT(128, 32, 128),
    GDN_VARIANT(128, 16, 64),   GDN_VARIANT(64, 64, 128),  GDN_VARIANT(64, 32, 64),
    GDN_VARIANT(64, 16, 32),    GDN_VARIANT(32, 32, 64),   GDN_VARIANT(32, 16, 32),
    GDN_VARIANT(16, 16, 32),
};
#undef GDN_VARIANT

const Variant *find_variant(int D, int W)
{
    for (const Variant &v : kVariants)
        if (v.D == D && v.W == W) return &v;
    return nullptr;
}

}  // namespace

bool plan_slab(int D, int B, int H_v, int group, int num_sms, StepPlan *plan)
{
    if (D != 16 && D != 32 && D != 64 && D != 128) return false;
    const long units = static_cast<long>(B) * H_v;
    // Fewest slabs that give every SM two CTAs, within an 8-CTA cluster and W >= 16.
    int best = 0;
    for (int nslab = 1; nslab <= 8; nslab *= 2) {
        const int W = D / nslab;
        if (W < 16 || nslab * group > 8 || !find_variant(D, W)) break;
        best = nslab;
        if (units * nslab >= 2L * num_sms) break;
    }
    // d = 128 from 64 units: two slabs a head measured fastest (B2 H32: 5.2 us a launch,
    // against 5.5 with four and 5.6 with eight; B1 is within 1% for 2, 4 or 8 slabs).
    if (D == 128 && units >= 64 && 2 * group <= 8) best = 2;
    if (best == 0) return false;
    const Variant *v = find_variant(D, D / best);
    plan->kind = StepPlan::kSlab;
    plan->D = D;
    plan->W = v->W;
    plan->nslab = best;
    plan->threads = v->NT;
    plan->cluster = best * group;
    plan->grid = static_cast<int>(units) * best;
    plan->name = v->name;
    return true;
}

// Long token loops (prefill on this kernel) run as one wave: every CTA holds its state
// slab for the whole sequence, so a grid larger than the GPU holds at once would run the
// loop twice over.  Halve the slab count of the regular plan until the grid fits.
bool plan_slab_one_wave(int D, int B, int H_v, int group, int num_sms, StepPlan *plan)
{
    if (!plan_slab(D, B, H_v, group, num_sms, plan)) return false;
    const long units = static_cast<long>(B) * H_v;
    while (plan->nslab > 1) {
        const Variant *v = find_variant(plan->D, plan->W);
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, v->fn, v->NT, 0) != cudaSuccess)
            per_sm = 1;
        if (units * plan->nslab <= static_cast<long>(per_sm) * num_sms) break;
        const int nslab = plan->nslab / 2;
        const Variant *w = find_variant(D, D / nslab);
        if (!w) break;
        plan->nslab = nslab;
        plan->W = w->W;
        plan->threads = w->NT;
        plan->cluster = nslab * group;
        plan->grid = static_cast<int>(units) * nslab;
        plan->name = w->name;
    }
    return true;
}

cudaError_t launch_slab(const StepPlan &plan, const StepArgs &a, bool pdl, cudaStream_t stream)
{
    const Variant *v = find_variant(plan.D, plan.W);
    if (!v) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.nslab, a.H_v, a.B);
    cfg.blockDim = dim3(plan.threads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    if (a.gate_lr) {
        const int gs = slab_gate_smem(plan.D, plan.W, a.gate_rank);
        if (a.T != 1 || !a.kda || a.gate_rank <= 0 || a.gate_rank % 8 || gs > kSlabGateSmemMax ||
            !a.w_fb || !a.w_gb || (reinterpret_cast<uintptr_t>(a.w_fb) & 15u) ||
            (reinterpret_cast<uintptr_t>(a.w_gb) & 15u))
            return cudaErrorInvalidValue;
        // static plus dynamic shared memory may pass the default 48 KB: opt in once per
        // device and variant (benign race: every writer sets the same value)
        static bool opted[64][sizeof(kVariants) / sizeof(kVariants[0])];
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        const size_t vi = static_cast<size_t>(v - kVariants);
        if (!opted[dev][vi]) {
            e = cudaFuncSetAttribute(v->fn_gates, cudaFuncAttributeMaxDynamicSharedMemorySize, kSlabGateSmemMax);
            if (e != cudaSuccess) return e;
            opted[dev][vi] = true;
        }
        cfg.dynamicSmemBytes = static_cast<size_t>(gs);
    }
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (plan.cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = plan.nslab;
        attr[n].val.clusterDim.y = a.group;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, a.gate_lr ? v->fn_gates : v->fn, a);
}

namespace {

struct WVariant {
    int NW;
    void (*fn)(StepArgs);
    const char *name;
};
const WVariant kWVariants[] = {
    {8, wstep_kernel<8>, "wstep<128,64>"},
    {16, wstep_kernel<16>, "wstep<128,128>"},
};

const WVariant *find_wvariant(int W)
{
    for (const WVariant &v : kWVariants)
        if (WCOL * v.NW == W) return &v;
    return nullptr;
}

}  // namespace

bool plan_wstep(int D, int B, int H_v, int group, int num_sms, StepPlan *plan)
{
    (void)num_sms;
    if (D != WD || group < 1 || group > 8) return false;
    const long units = static_cast<long>(B) * H_v;
    // Below 128 units the column-slab kernel keeps the shorter chain (B1 H32: 4.4
    // against 5.8 us a launch; B2: 5.2 against 6.8).  From 128 units two 64-column
    // slabs a head measured fastest (B4 H32: 8.8 us, against 10.1 on the slab kernel
    // and 9.1 with whole heads; B8: 17.3 against 20.1).
    if (units < 128) return false;
    const int best = 2 * group <= 8 ? 2 : 1;
    const WVariant *v = find_wvariant(D / best);
    plan->kind = StepPlan::kWarp;
    plan->D = D;
    plan->W = D / best;
    plan->nslab = best;
    plan->threads = v->NW * 32;
    plan->cluster = best * group;
    plan->grid = static_cast<int>(units) * best;
    plan->name = v->name;
    return true;
}

cudaError_t launch_wstep(const StepPlan &plan, const StepArgs &a, bool pdl, cudaStream_t stream)
{
    if (a.gate_lr) return cudaErrorInvalidValue;  // in-kernel gates: slab kernel only
    const WVariant *v = find_wvariant(plan.W);
    if (!v || plan.D != WD) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.nslab, a.H_v, a.B);
    cfg.blockDim = dim3(v->NW * 32, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (plan.cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = plan.nslab;
        attr[n].val.clusterDim.y = a.group;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, v->fn, a);
}

unsigned int take_step_error()
{
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_step_error, sizeof(v)) != cudaSuccess) return ~0u;
    if (v && cudaMemcpyToSymbol(g_step_error, &zero, sizeof(zero)) != cudaSuccess) return ~0u;
    return v;
}

}  // namespace gdn
