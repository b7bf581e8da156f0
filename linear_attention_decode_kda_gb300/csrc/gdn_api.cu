// C ABI of the KDA / Gated DeltaNet step: argument validation and dispatch.
// Every check runs on the host before anything is queued; nothing here
// allocates, copies or synchronises.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "gdn.h"
#include "gdn_internal.h"
#include "gdn_prefill.h"

namespace {

constexpr int kMaxDevices = 64;
int g_num_sms[kMaxDevices];  // 0 = not queried yet; benign race: every writer stores the same value

int num_sms_current()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    if (g_num_sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 0;
        g_num_sms[dev] = n;
    }
    return g_num_sms[dev];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape checks shared by every entry point (T is checked by the caller).
gdn_status_t check_shape(const gdn_shape_t *s)
{
    if (!s) return GDN_ERR_NULL;
    if (s->B < 0 || s->T < 0 || s->H_qk <= 0 || s->H_v <= 0 || s->d_k <= 0 || s->d_v <= 0)
        return GDN_ERR_SHAPE;
    if (s->H_v % s->H_qk != 0) return GDN_ERR_SHAPE;
    if (s->B > 65535 || s->H_v > 65535) return GDN_ERR_SHAPE;
    if (s->gate_mode != GDN_GATE_PER_HEAD && s->gate_mode != GDN_GATE_PER_CHANNEL &&
        s->gate_mode != GDN_GATE_LOWER_BOUND)
        return GDN_ERR_SHAPE;
    if ((s->in_dtype != GDN_F32 && s->in_dtype != GDN_BF16) ||
        (s->out_dtype != GDN_F32 && s->out_dtype != GDN_BF16))
        return GDN_ERR_SHAPE;
    if (s->flags & ~(GDN_FLAG_PDL | GDN_FLAG_SIGMOID_GATE)) return GDN_ERR_SHAPE;
    if (!(s->q_scale > 0.0f) || !(s->eps_l2 >= 0.0f) || !(s->eps_norm >= 0.0f))
        return GDN_ERR_SHAPE;
    if (s->conv_K != 4) return GDN_ERR_UNSUPPORTED;
    if (s->d_k != s->d_v) return GDN_ERR_UNSUPPORTED;
    const long C = 2L * s->H_qk * s->d_k + static_cast<long>(s->H_v) * s->d_v;
    if (C > (1L << 30)) return GDN_ERR_SHAPE;
    return GDN_OK;
}

bool aligned(const void *p, unsigned bytes) { return (reinterpret_cast<uintptr_t>(p) % bytes) == 0; }

// Vector-accessed buffers (state, conv_w, out) need 16 bytes; the rest their element size.
// `out` may be NULL only where the entry point allows it.
gdn_status_t check_tensors(const gdn_shape_t *s, const gdn_tensors_t *t, bool out_optional = false)
{
    if (!t) return GDN_ERR_NULL;
    const void *req[] = {t->qkv, t->f, t->beta, t->z, t->conv_w, t->A_log, t->dt_bias,
                         t->norm_w, t->conv_state, t->state};
    for (const void *p : req)
        if (!p) return GDN_ERR_NULL;
    if (!t->out && !out_optional) return GDN_ERR_NULL;
    const unsigned ib = s->in_dtype == GDN_BF16 ? 2u : 4u;
    if (!aligned(t->qkv, ib) || !aligned(t->f, ib) || !aligned(t->beta, ib) ||
        !aligned(t->z, ib) || !aligned(t->A_log, 4) || !aligned(t->dt_bias, 4) ||
        !aligned(t->norm_w, 4) || !aligned(t->conv_state, 4) || !aligned16(t->conv_w) ||
        !aligned16(t->state) || !aligned16(t->out))
        return GDN_ERR_ALIGN;
    return GDN_OK;
}

gdn::StepArgs step_args(const gdn_shape_t *s, const gdn_tensors_t *t)
{
    gdn::StepArgs a = {};
    a.qkv = t->qkv;
    a.f = t->f;
    a.beta = t->beta;
    a.z = t->z;
    a.conv_w = t->conv_w;
    a.A_log = t->A_log;
    a.dt_bias = t->dt_bias;
    a.norm_w = t->norm_w;
    a.state_in = t->state;
    a.conv_in = t->conv_state;
    a.out = t->out;
    a.B = s->B;
    a.T = s->T;
    a.Ts = s->T;
    a.H_qk = s->H_qk;
    a.H_v = s->H_v;
    a.C = 2 * s->H_qk * s->d_k + s->H_v * s->d_v;
    a.group = s->H_v / s->H_qk;
    a.kda = s->gate_mode != GDN_GATE_PER_HEAD;
    a.lb_gate = s->gate_mode == GDN_GATE_LOWER_BOUND;
    a.sig_gate = (s->flags & GDN_FLAG_SIGMOID_GATE) != 0;
    a.in_bf16 = s->in_dtype == GDN_BF16;
    a.out_bf16 = s->out_dtype == GDN_BF16;
    a.q_scale = s->q_scale;
    a.eps_l2 = s->eps_l2;
    a.eps_norm = s->eps_norm;
    return a;
}

bool plan_for(const gdn_shape_t *s, gdn::StepPlan *plan)
{
    const int sms = num_sms_current();
    return gdn::plan_step(s->d_k, s->B, s->H_v, s->H_v / s->H_qk, sms > 0 ? sms : 148, plan);
}

// Scratch of gdn_prefill_chunked_static, for callers that cannot allocate:
// a module-scope device array, reserved when the module loads in a context.
// Its device address is looked up once per device and context: a context torn
// down and made again (cudaDeviceReset) reloads the module at a new address,
// so the cached address is kept together with the context it belongs to.
// Writers race benignly (every writer stores the same pair).
static __device__ __align__(256) unsigned char g_prefill_scratch[GDN_PREFILL_STATIC_SCRATCH_BYTES];
struct ScratchAddr {
    CUcontext ctx;
    void *ptr;
};
ScratchAddr g_scratch_addr[kMaxDevices];

PFN_cuCtxGetCurrent_v4000 ctx_getter()
{
    static PFN_cuCtxGetCurrent_v4000 fn = nullptr;  // benign race: same value
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    }
    return fn;
}

void *static_scratch()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    PFN_cuCtxGetCurrent_v4000 get_ctx = ctx_getter();
    if (!get_ctx) return nullptr;
    ScratchAddr &c = g_scratch_addr[dev];
    CUcontext ctx = nullptr;  // NULL until the runtime has made a context current
    if (get_ctx(&ctx) == CUDA_SUCCESS && ctx && c.ctx == ctx && c.ptr) return c.ptr;
    void *p = nullptr;  // the lookup makes the device's primary context current if needed
    if (cudaGetSymbolAddress(&p, g_prefill_scratch) != cudaSuccess) return nullptr;
    if (get_ctx(&ctx) != CUDA_SUCCESS || !ctx) return nullptr;
    c.ptr = p;
    c.ctx = ctx;
    return p;
}

// The prefill after its checks: with snapshot tails when state_hist or conv_hist is set.
gdn_status_t prefill_call(const gdn_shape_t *s, const gdn_tensors_t *t, void *workspace,
                          cudaStream_t stream)
{
    gdn::StepArgs a = step_args(s, t);
    a.state_out = t->state;
    a.conv_out = t->conv_state;
    const int sms = num_sms_current();
    if (t->state_hist || t->conv_hist) {
        a.state_hist = t->state_hist;
        a.conv_hist = t->conv_hist;
        return gdn::run_prefill_snapshots(*s, a, workspace, sms > 0 ? sms : 148, stream);
    }
    return gdn::run_prefill(*s, a, workspace, sms > 0 ? sms : 148, stream);
}

gdn_status_t run_step(const gdn_shape_t *s, const gdn::StepArgs &a, cudaStream_t stream)
{
    gdn::StepPlan plan;
    if (!plan_for(s, &plan)) return GDN_ERR_UNSUPPORTED;
    const int sms = num_sms_current();
    cudaError_t e = gdn::launch_step(plan, a, (s->flags & GDN_FLAG_PDL) != 0, sms > 0 ? sms : 148,
                                     stream);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

extern "C" {

gdn_status_t gdn_decode_step(const gdn_shape_t *s, const gdn_tensors_t *t, gdn_stream_t stream)
{
    gdn_status_t rc = check_shape(s);
    if (rc != GDN_OK) return rc;
    if (s->T != 1) return GDN_ERR_SHAPE;
    rc = check_tensors(s, t);
    if (rc != GDN_OK) return rc;
    gdn::StepPlan plan;
    if (!plan_for(s, &plan)) return GDN_ERR_UNSUPPORTED;
    if (s->B == 0) return GDN_OK;
    gdn::StepArgs a = step_args(s, t);
    a.state_out = t->state;
    a.conv_out = t->conv_state;
    return run_step(s, a, reinterpret_cast<cudaStream_t>(stream));
}

gdn_status_t gdn_verify_T(const gdn_shape_t *s, const gdn_tensors_t *t, gdn_stream_t stream)
{
    gdn_status_t rc = check_shape(s);
    if (rc != GDN_OK) return rc;
    if (s->T < 1 || s->T > 4) return GDN_ERR_SHAPE;
    rc = check_tensors(s, t);
    if (rc != GDN_OK) return rc;
    if ((t->state_hist && !aligned16(t->state_hist)) || (t->conv_hist && !aligned(t->conv_hist, 4)))
        return GDN_ERR_ALIGN;
    gdn::StepPlan plan;
    if (!plan_for(s, &plan)) return GDN_ERR_UNSUPPORTED;
    if (s->B == 0) return GDN_OK;
    gdn::StepArgs a = step_args(s, t);
    a.state_hist = t->state_hist;
    a.conv_hist = t->conv_hist;
    return run_step(s, a, reinterpret_cast<cudaStream_t>(stream));
}

gdn_status_t gdn_commit_accepted(const gdn_shape_t *s, const gdn_tensors_t *t, const int32_t *accepted,
                                 gdn_stream_t stream)
{
    gdn_status_t rc = check_shape(s);
    if (rc != GDN_OK) return rc;
    if (s->T < 1 || s->T > 4) return GDN_ERR_SHAPE;
    rc = check_tensors(s, t, true);
    if (rc != GDN_OK) return rc;
    if (accepted && !aligned(accepted, 4)) return GDN_ERR_ALIGN;
    gdn::StepPlan plan;
    if (!plan_for(s, &plan)) return GDN_ERR_UNSUPPORTED;
    if (s->B == 0) return GDN_OK;
    gdn::StepArgs a = step_args(s, t);
    a.state_out = t->state;
    a.conv_out = t->conv_state;
    a.accepted = accepted;
    return run_step(s, a, reinterpret_cast<cudaStream_t>(stream));
}

size_t gdn_prefill_workspace_bytes(const gdn_shape_t *s)
{
    if (check_shape(s) != GDN_OK || s->T < 1) return 0;
    return gdn::prefill_workspace_bytes(*s);
}

gdn_status_t gdn_prefill_chunked(const gdn_shape_t *s, const gdn_tensors_t *t, void *workspace,
                                 size_t workspace_bytes, gdn_stream_t stream)
{
    gdn_status_t rc = check_shape(s);
    if (rc != GDN_OK) return rc;
    if (s->T < 1) return GDN_ERR_SHAPE;
    rc = check_tensors(s, t);
    if (rc != GDN_OK) return rc;
    if (s->chunk <= 0) return GDN_ERR_SHAPE;
    if ((t->state_hist && !aligned16(t->state_hist)) || (t->conv_hist && !aligned(t->conv_hist, 4)))
        return GDN_ERR_ALIGN;
    const size_t need = gdn::prefill_workspace_bytes(*s);
    if (workspace_bytes < need || (need > 0 && !workspace)) return GDN_ERR_WORKSPACE;
    if (workspace && !aligned16(workspace)) return GDN_ERR_ALIGN;
    if (s->B == 0) return GDN_OK;
    return prefill_call(s, t, workspace, reinterpret_cast<cudaStream_t>(stream));
}

gdn_status_t gdn_prefill_chunked_static(const gdn_shape_t *s, const gdn_tensors_t *t,
                                        gdn_stream_t stream)
{
    gdn_status_t rc = check_shape(s);
    if (rc != GDN_OK) return rc;
    if (s->T < 1) return GDN_ERR_SHAPE;
    rc = check_tensors(s, t);
    if (rc != GDN_OK) return rc;
    if (s->chunk <= 0) return GDN_ERR_SHAPE;
    if ((t->state_hist && !aligned16(t->state_hist)) || (t->conv_hist && !aligned(t->conv_hist, 4)))
        return GDN_ERR_ALIGN;
    const size_t need = gdn::prefill_workspace_bytes(*s);
    if (need > GDN_PREFILL_STATIC_SCRATCH_BYTES) return GDN_ERR_WORKSPACE;
    if (s->B == 0) return GDN_OK;
    void *ws = nullptr;
    if (need > 0) {
        ws = static_scratch();
        if (!ws) return GDN_ERR_CUDA;
    }
    // no clearing: the intra-chunk kernel writes every scratch word the state kernel uses
    return prefill_call(s, t, ws, reinterpret_cast<cudaStream_t>(stream));
}

size_t gdn_layer_workspace_bytes(const gdn_shape_t *s, const gdn_layer_weights_t *w)
{
    if (check_shape(s) != GDN_OK || !w || w->rank <= 0 || s->B < 0) return 0;
    return static_cast<size_t>(s->B) * 2 * w->rank * sizeof(float);
}

gdn_status_t gdn_layer_decode(const gdn_shape_t *s, const gdn_layer_weights_t *w, const void *x,
                              float *x_out, const gdn_tensors_t *t, void *workspace,
                              size_t workspace_bytes, gdn_stream_t stream)
{
    gdn_status_t rc = check_shape(s);
    if (rc != GDN_OK) return rc;
    if (s->T != 1 || s->gate_mode == GDN_GATE_PER_HEAD || s->in_dtype != GDN_F32 ||
        s->out_dtype != GDN_F32)
        return GDN_ERR_SHAPE;
    rc = check_tensors(s, t);
    if (rc != GDN_OK) return rc;
    if (!w || !x || !x_out || !w->w_qkv || !w->w_fa || !w->w_fb || !w->w_ga || !w->w_gb ||
        !w->w_beta || !w->w_o)
        return GDN_ERR_NULL;
    if (w->d_model <= 0 || w->rank <= 0 || w->d_model % 8 || w->rank % 8) return GDN_ERR_SHAPE;
    const void *wp[] = {w->w_qkv, w->w_fa, w->w_fb, w->w_ga, w->w_gb, w->w_beta, w->w_o, x,
                        t->qkv, t->f, t->beta, t->z, t->out};
    for (const void *p : wp)
        if (!aligned16(p)) return GDN_ERR_ALIGN;
    if (!aligned(x_out, 4)) return GDN_ERR_ALIGN;
    const size_t need = gdn_layer_workspace_bytes(s, w);
    if (workspace_bytes < need || (need > 0 && !workspace)) return GDN_ERR_WORKSPACE;
    if (workspace && !aligned16(workspace)) return GDN_ERR_ALIGN;
    gdn::StepPlan plan;
    if (!plan_for(s, &plan)) return GDN_ERR_UNSUPPORTED;
    if (s->B == 0) return GDN_OK;
    const int B = s->B, D = w->d_model, R = w->rank, C = 2 * s->H_qk * s->d_k + s->H_v * s->d_v;
    const int HK = s->H_v * s->d_k, HV = s->H_v * s->d_v;
    float *lr = static_cast<float *>(workspace);  // [B][2R]: f_a, then g_a
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float *qkv = static_cast<float *>(const_cast<void *>(t->qkv));
    float *f = static_cast<float *>(const_cast<void *>(t->f));
    float *beta = static_cast<float *>(const_cast<void *>(t->beta));
    float *z = static_cast<float *>(const_cast<void *>(t->z));
    const gdn::ProjSlotDesc in[4] = {
        {w->w_qkv, x, qkv, C, D, D, C, 1},
        {w->w_fa, x, lr, R, D, D, 2 * R, 1},
        {w->w_ga, x, lr + R, R, D, D, 2 * R, 1},
        {w->w_beta, x, beta, s->H_v, D, D, s->H_v, 1},
    };
    const gdn::ProjSlotDesc gate[2] = {
        {w->w_fb, lr, f, HK, R, 2 * R, HK, 0},
        {w->w_gb, lr + R, z, HV, R, 2 * R, HV, 0},
    };
    const gdn::ProjSlotDesc out[1] = {{w->w_o, t->out, x_out, D, HV, HV, D, 0}};
    for (const auto &d : in)
        if (!gdn::proj_slot_ok(d)) return GDN_ERR_ALIGN;
    for (const auto &d : gate)
        if (!gdn::proj_slot_ok(d)) return GDN_ERR_ALIGN;
    if (!gdn::proj_slot_ok(out[0])) return GDN_ERR_ALIGN;
    if (gdn::launch_proj(in, 4, B, st, false) != cudaSuccess) return GDN_ERR_CUDA;
    gdn::StepArgs a = step_args(s, t);
    a.state_out = t->state;
    a.conv_out = t->conv_state;
    // On the column-slab kernel the low-rank gates' second products run inside the
    // step (each CTA from its head's W_fb rows and its columns' W_gb rows), which saves
    // a launch and its dependency on the critical path; otherwise the gate pair is a
    // projection launch of its own.
    if (plan.kind == gdn::StepPlan::kSlab &&
        gdn::slab_gate_smem(plan.D, plan.W, R) <= gdn::kSlabGateSmemMax) {
        a.gate_lr = lr;
        a.w_fb = w->w_fb;
        a.w_gb = w->w_gb;
        a.gate_rank = R;
        a.gate_f = f;
        a.gate_z = z;
    } else if (gdn::launch_proj(gate, 2, B, st, true) != cudaSuccess) {
        return GDN_ERR_CUDA;
    }
    // The step overlaps its prologue with the projections before it, which write only
    // the rows it reads after its dependency wait.
    gdn_shape_t sp = *s;
    sp.flags |= GDN_FLAG_PDL;
    rc = run_step(&sp, a, st);
    if (rc != GDN_OK) return rc;
    return gdn::launch_proj(out, 1, B, st, true) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

const char *gdn_status_string(gdn_status_t status)
{
    switch (status) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_NULL: return "GDN_ERR_NULL: a required pointer is NULL";
    case GDN_ERR_ALIGN: return "GDN_ERR_ALIGN: a pointer is misaligned";
    case GDN_ERR_SHAPE: return "GDN_ERR_SHAPE: invalid sizes";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: no kernel instance for these sizes";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE: workspace missing or too small";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA: the CUDA runtime refused a launch";
    case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT: a bounded device wait gave up";
    }
    return "unknown gdn_status_t";
}

gdn_status_t gdn_device_status(void)
{
    const unsigned int e = gdn::take_stream_error(), p = gdn::take_prefill_error(),
                       q = gdn::take_step_error(), r = gdn::take_kda_prefill_error(),
                       w = gdn::take_proj_error(), c = gdn::take_c64_error();
    if (e == ~0u || p == ~0u || q == ~0u || r == ~0u || w == ~0u || c == ~0u) return GDN_ERR_CUDA;
    return (e | p | q | r | w | c) ? GDN_ERR_TIMEOUT : GDN_OK;
}

const char *gdn_kernel_variant(const gdn_shape_t *s, int op)
{
    if (check_shape(s) != GDN_OK) return nullptr;
    if (op == 2) return gdn::prefill_variant(*s, num_sms_current());
    gdn::StepPlan plan;
    if ((op != 0 && op != 1) || !plan_for(s, &plan)) return nullptr;
    return plan.name;
}

}  // extern "C"
