// workspace.h -- internal (not part of the C ABI): the layout of the split
// tail's workspace, for code in this library that manages a workspace of
// its own.
#pragma once

#include <cstddef>
#include <cstdint>

#include "gemm.h"

namespace gb300 {

// For a gemm_run_workspace call with these arguments (and a large enough
// workspace): the bytes of counter words at the start of the workspace, which
// must read as zero for this call's launch, and the total bytes the call
// needs (both 0 when the plan does not split).  The rest of the workspace
// holds FP32 partials, each written before it is read.  Returns the argument
// errors of gemm_workspace_size.
__attribute__((visibility("hidden"))) int split_workspace_layout(
    int64_t M, int64_t N, int64_t K, int dtype, int b_layout, const gemm_options_t* opts,
    size_t* counter_bytes, size_t* total_bytes);

}  // namespace gb300
