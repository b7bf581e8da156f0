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
    void *out;                   // [B,T,H_v,D]
    float *state_hist;           // [T,B,H_v,D,D] or NULL
    float *conv_hist;            // [T,B,K-1,C] or NULL
    int B, T, H_qk, H_v, C;
    int group;                   // H_v / H_qk
    int kda, in_bf16, out_bf16;
    float q_scale, eps_l2, eps_norm;
};

// One launch configuration of the step kernel.
struct StepPlan {
    int D = 0, W = 0, nslab = 0, threads = 0, cluster = 1;
    const char *name = nullptr;
};

// Chooses the column-slab width for B*H_v head units on a GPU with `num_sms` SMs.
bool plan_step(int D, int B, int H_v, int group, int num_sms, StepPlan *plan);

// Queues the step kernel.  pdl: programmatic dependent launch attribute.
cudaError_t launch_step(const StepPlan &plan, const StepArgs &a, bool pdl, cudaStream_t stream);

}  // namespace gdn
