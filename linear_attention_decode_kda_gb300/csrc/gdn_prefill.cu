// Prefill: T tokens per sequence, state and conv window advanced in place.
// This version runs the tokens through the recurrent step kernel (the state
// stays in registers across all T tokens).
#include "gdn_prefill.h"

namespace gdn {

size_t prefill_workspace_bytes(const gdn_shape_t &) { return 0; }

const char *prefill_variant(const gdn_shape_t &s, int num_sms)
{
    StepPlan plan;
    if (!plan_step(s.d_k, s.B, s.H_v, s.H_v / s.H_qk, num_sms > 0 ? num_sms : 148, &plan))
        return nullptr;
    return plan.name;
}

gdn_status_t run_prefill(const gdn_shape_t &s, const StepArgs &a, void *, int num_sms,
                         cudaStream_t stream)
{
    StepPlan plan;
    if (!plan_step(s.d_k, s.B, s.H_v, s.H_v / s.H_qk, num_sms, &plan)) return GDN_ERR_UNSUPPORTED;
    cudaError_t e = launch_step(plan, a, (s.flags & GDN_FLAG_PDL) != 0, num_sms, stream);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace gdn
