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

// Reads and clears the chunked prefill kernel's device error word (synchronous).
unsigned int take_prefill_error();

}  // namespace gdn
