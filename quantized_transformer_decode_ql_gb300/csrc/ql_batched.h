// The batch 3-32 GEMV's profiling entry point (ql_batched.cu).
#pragma once

#include "ql_internal.h"

namespace ql {

// batched_gemv_launch, with globaltimer stamps of the merge launch written to merge_trace when
// it is not null: [num_SMs CTAs][4] = 0 start, 1 past the wait on the GEMV, 2 the CTA's
// items done, 3 end (QL_OPT_MERGE_TRACE). A null merge_trace is batched_gemv_launch itself.
int batched_gemv_launch_traced(const StreamGemvArgs& a, unsigned long long* merge_trace, cudaStream_t s, bool pdl);

constexpr int kMergeTraceWords = 4;   // merge trace entries per CTA

}  // namespace ql
