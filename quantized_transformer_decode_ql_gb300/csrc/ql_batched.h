// Internal entry points of the batch 3-32 GEMV's profiling form (ql_batched.cu) and of the q4_0
// GEMM for prompt chunks (ql_gemm.cu).
#pragma once

#include <cuda.h>   // CUtensorMap

#include "ql_internal.h"

namespace ql {

// batched_gemv_launch, with globaltimer stamps of the merge launch written to merge_trace when
// it is not null: [num_SMs CTAs][4] = 0 start, 1 past the wait on the GEMV, 2 the CTA's
// items done, 3 end (QL_OPT_MERGE_TRACE). A null merge_trace is batched_gemv_launch itself.
int batched_gemv_launch_traced(const StreamGemvArgs& a, unsigned long long* merge_trace, cudaStream_t s, bool pdl);

constexpr int kMergeTraceWords = 4;   // merge trace entries per CTA

// Prompt chunks (ql_prefill_chunk): up to kPrefillGemvMax tokens through the decode step's GEMVs,
// above it through the GEMM; at most kPrefillMax tokens per chunk.
constexpr int kPrefillGemvMax = 32;
constexpr int kPrefillMax = 256;

// Tensor maps (the driver's encoder, QL_ECUDA if it is unavailable or refuses the layout):
// the tile stream of M as [tile][unit][144 x 8 B] with boxes of 8 tiles x 1 unit; and a
// row-major f16 matrix [outer][inner] (16-byte aligned base, inner % 8 == 0) with boxes of
// box_outer rows x box_inner elements, reads past the matrix returning zero; swizzle128: the
// box lands with the 128-byte swizzle (box_inner * 2 == 128, a 1024-byte aligned destination).
int q4_stream_tensor_map(const PMat& M, CUtensorMap* map);
int f16_rows_tensor_map(const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer,
                        CUtensorMap* map, bool swizzle128);

// The prompt GEMM (ql_gemm.cu): y[t][r] = sum_k W[r][k] x16[t][k] for t < T over the tile stream
// copy of W (M.stream), with the epilogue QL_EPI_NONE (f32 y), QL_EPI_ADD_RESIDUAL (f32 y +=) or
// QL_EPI_SILU_MUL (f16 y [T][rows / 2] = SiLU(gate) * up, M packed for it); ld is y's row pitch
// in elements. x16: f16 [T][K], 16-byte aligned.
// part (optional, part_bytes): scratch for splitting K over CTAs when the matrix has few row
// blocks (then a second kernel adds the parts in order); null: no split.
struct GemmArgs {
    PMat M;
    int T;
    const __half* x16;
    void* y;
    int ld;
    int epi;
    float* part;
    size_t part_bytes;
};
int gemm_tc_launch(const GemmArgs& a, cudaStream_t s, bool pdl);

// RMSNorm of T columns: xn[t] = f16(x[t] / rms(x[t]) * w), x f32 [T][cols] (ql_batched.cu).
int rms_norm_launch(const float* x, int cols, float eps, const float* w, __half* xn, int T, cudaStream_t s, bool pdl);

}  // namespace ql
