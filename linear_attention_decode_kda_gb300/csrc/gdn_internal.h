// Internal interface between the C ABI (gdn_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gdn {

// Arguments of the recurrent step kernel (decode, verify, recurrent tail of prefill).
struct StepArgs {
    const void *qkv, *f, *beta, *z;
    const float *conv_w, *A_log, *dt_bias, *norm_w;
    const float *state_in;       // [B,H_v,D,D] state read at the first token
    float *state_out;            // commit: final state (may equal state_in); else NULL
    const float *conv_in;        // [B,K-1,C] conv window read at the first token
    float *conv_out;             // commit: final window (may equal conv_in); else NULL
    void *out;                   // [B,T,H_v,D], or NULL (commit without outputs)
    float *state_hist;           // [T,B,H_v,D,D] or NULL
    float *conv_hist;            // [T,B,K-1,C] or NULL
    const int32_t *accepted;     // [B]: tokens taken per sequence (clamped to 0..T), or NULL for T
    int B, T, H_qk, H_v, C;
    int Ts;                      // token stride of the [B, Ts, ...] rows: T, or more for a part of a call
    int group;                   // H_v / H_qk
    int kda;                     // one decay per key channel (both per-channel gate forms)
    int lb_gate;                 // lower-bound gate: A_log = scale a, dt_bias[h] = bound lb
    int sig_gate;                // output gate sigmoid(z) instead of silu(z)
    int in_bf16, out_bf16;
    float q_scale, eps_l2, eps_norm;
    // Low-rank gates inside the column-slab kernel (a layer's decode, T = 1, per-channel
    // decay): f[b,h,:] = W_fb[h D .. h D + D) lr[b, 0:R] and z[b,h,:] likewise from W_gb
    // and lr[b, R:2R]; lr is [B][2R] fp32, W_fb and W_gb [H_v D][R] bf16 (16-byte
    // aligned, R a multiple of 8).  NULL: f and z are read as rows.  Only the slab
    // kernel takes them (slab_gate_smem bytes of dynamic shared memory): each slab
    // computes f for its own W key channels and hands them to the head's other slabs
    // through the cluster.
    const float *gate_lr;
    const void *w_fb, *w_gb;
    int gate_rank;
    float *gate_f, *gate_z;  // the in-kernel gates' f and z also stored as rows (fp32), or NULL
};

// Dynamic shared memory of the slab kernel's in-kernel gates: the W_fb rows of the
// slab's key channels and the W_gb rows of its value columns (each padded by 16 bytes),
// and the lr row.
inline int slab_gate_smem(int D, int W, int R)
{
    (void)D;
    return 2 * W * (2 * R + 16) + 8 * R;
}
// at most this much (the kernels' static shared memory is under 12 KB; the opt-in
// limit is 227 KB): past it the gate pair runs as a launch of its own
constexpr int kSlabGateSmemMax = 96 * 1024;

// One launch configuration of the step kernels.
struct StepPlan {
    enum Kind { kSlab, kStream, kWarp } kind = kSlab;
    int D = 0, W = 0, nslab = 0, threads = 0, cluster = 1, grid = 0;
    const char *name = nullptr;
};

// Column-slab kernel (gdn_step.cu): any unit count, d in {16, 32, 64, 128}.
bool plan_slab(int D, int B, int H_v, int group, int num_sms, StepPlan *plan);
cudaError_t launch_slab(const StepPlan &plan, const StepArgs &a, bool pdl, cudaStream_t stream);
// The slab plan for long token loops: as plan_slab, with fewer slabs until the grid is
// resident at once.
bool plan_slab_one_wave(int D, int B, int H_v, int group, int num_sms, StepPlan *plan);

// Warp-column kernel (gdn_step.cu): d = 128, every reduction of a token inside a
// warp, 64 or 128 value columns a CTA; planned from 128 (sequence, head) units.
bool plan_wstep(int D, int B, int H_v, int group, int num_sms, StepPlan *plan);
cudaError_t launch_wstep(const StepPlan &plan, const StepArgs &a, bool pdl, cudaStream_t stream);

// Persistent TMA-pipelined kernel (gdn_stream.cu): d = 128, ungrouped heads,
// more than 64 (sequence, head) units.
bool plan_stream(int D, int B, int H_v, int group, int num_sms, StepPlan *plan);
// True when every buffer meets the streaming kernel's 16-byte chunk rules.
bool stream_eligible(const StepArgs &a);
cudaError_t launch_stream(const StepPlan &plan, const StepArgs &a, bool pdl, cudaStream_t stream);

// Weight-streaming projections around the step (gdn_proj.cu): per slot,
// y[b][n] = sum_k x[b][k] w[n][k] with w bf16 [N][K] (row-major, 16-byte aligned,
// K % 8 == 0), x fp32 or bf16 rows of stride ldx (16-byte aligned), y fp32 rows
// of stride ldy.  One launch covers up to kMaxProjSlots slots.
constexpr int kMaxProjSlots = 4;
constexpr int kProjTcMinBatch = 16;  // from this batch up the products run on tcgen05 (K % 64 == 0)
struct ProjSlotDesc {
    const void *w;
    const void *x;
    float *y;
    int N, K, ldx, ldy, x_bf16;
};
bool proj_slot_ok(const ProjSlotDesc &d);
// Launched with programmatic dependent launch (the kernels read activations and write
// outputs after their dependency wait).  prefetch: below the tensor-core batch, ask L2
// for the weights before that wait, for a launch that follows another kernel it can
// overlap (the gate pair and the output projection of a layer).
cudaError_t launch_proj(const ProjSlotDesc *slots, int nslot, int B, cudaStream_t stream, bool prefetch);
unsigned int take_proj_error();

// Read and clear the step kernels' device error words (synchronous).
unsigned int take_stream_error();
unsigned int take_step_error();

// The plan for B*H_v units on a GPU with `num_sms` SMs.  Decode and verify of
// the same (B, H_v) always get the same plan, so their per-token arithmetic
// is identical.
inline bool plan_step(int D, int B, int H_v, int group, int num_sms, StepPlan *plan)
{
    return plan_stream(D, B, H_v, group, num_sms, plan) ||
           plan_wstep(D, B, H_v, group, num_sms, plan) ||
           plan_slab(D, B, H_v, group, num_sms, plan);
}

// Queues the planned kernel; a streaming plan whose buffers miss the 16-byte
// chunk rules runs on the warp-column (d = 128) or column-slab kernel instead.
inline cudaError_t launch_step(const StepPlan &plan, const StepArgs &a, bool pdl, int num_sms,
                               cudaStream_t stream)
{
    if (plan.kind == StepPlan::kStream) {
        if (stream_eligible(a)) return launch_stream(plan, a, pdl, stream);
        StepPlan other;
        if (plan_wstep(plan.D, a.B, a.H_v, a.group, num_sms, &other))
            return launch_wstep(other, a, pdl, stream);
        if (!plan_slab(plan.D, a.B, a.H_v, a.group, num_sms, &other)) return cudaErrorInvalidValue;
        return launch_slab(other, a, pdl, stream);
    }
    if (plan.kind == StepPlan::kWarp) return launch_wstep(plan, a, pdl, stream);
    return launch_slab(plan, a, pdl, stream);
}

}  // namespace gdn
