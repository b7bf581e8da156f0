// Internal interface of the prefill path.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "gdn.h"
#include "gdn_internal.h"

namespace gdn {

// Device workspace bytes gdn_prefill_chunked needs for this shape.
size_t prefill_workspace_bytes(const gdn_shape_t &s);

// Name of the prefill variant for this shape, or nullptr.
const char *prefill_variant(const gdn_shape_t &s, int num_sms);

// Queues the prefill.  `a` carries the tensors with state_out / conv_out set.
gdn_status_t run_prefill(const gdn_shape_t &s, const StepArgs &a, void *workspace, int num_sms,
                         cudaStream_t stream);

// The prefill with snapshot tails: the first T - n tokens (n = min(T, 4)) as
// run_prefill, then the last n on the recurrent step kernel, which writes
// a.state_hist / a.conv_hist after each of them and leaves the final state and
// window in place.  `a` carries the tensors with state_out / conv_out set.
gdn_status_t run_prefill_snapshots(const gdn_shape_t &s, const StepArgs &a, void *workspace,
                                   int num_sms, cudaStream_t stream);

// Reads and clears the chunked prefill kernel's device error word (synchronous).
unsigned int take_prefill_error();

// Two-kernel chunked form (gdn_kda_prefill.cu): d = 128, any gate, T > 4.
bool kda_chunk_shape(const gdn_shape_t &s);
// The kernels' pointer rule beyond the ABI's: z 16-byte aligned (else the recurrent kernel runs).
bool kda_chunk_pointers_ok(const StepArgs &a);
size_t kda_chunk_workspace_bytes(const gdn_shape_t &s);
// Queues the intra-chunk kernel, then the state kernel; `workspace` holds
// kda_chunk_workspace_bytes(s) bytes, 16-byte aligned.
cudaError_t launch_kda_chunked(const StepArgs &a, void *workspace, cudaStream_t stream);
unsigned int take_kda_prefill_error();

// 64-token chunked form on tcgen05 (gdn_c64_prefill.cu): per-head decay, d = 128, bf16 rows,
// shape->chunk == 64; no workspace.
bool c64_shape(const gdn_shape_t &s);
// Its pointer rule beyond the ABI's: qkv and z 16-byte aligned (they arrive by TMA).
bool c64_pointers_ok(const StepArgs &a);
cudaError_t launch_c64(const StepArgs &a, cudaStream_t stream);
unsigned int take_c64_error();

}  // namespace gdn
