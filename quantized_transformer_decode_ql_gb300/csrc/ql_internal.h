// Internal declarations shared by the libql translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <string>

#include "../../include/ql.h"

namespace ql {

// ---------------------------------------------------------------- errors (host)
int set_error(int status, const std::string& msg);
int cuda_error(cudaError_t e, const char* what);

#define QL_TRY_CUDA(call)                                                    \
    do {                                                                     \
        cudaError_t e_ = (call);                                             \
        if (e_ != cudaSuccess) return ::ql::cuda_error(e_, #call);           \
    } while (0)

#define QL_REQUIRE(cond, msg)                                                \
    do {                                                                     \
        if (!(cond)) return ::ql::set_error(QL_EINVAL, msg);                 \
    } while (0)

// ---------------------------------------------------------------- device error record
// First out-of-range event seen by any kernel on a device. Kernels record with
// record_device_error() and skip the access; the host reads it in ql_check_device_error.
struct DevError {
    int code;      // nonzero once something was recorded
    int where;     // which kernel (DevErrWhere)
    long long index;
    long long value;
};
enum DevErrWhere {
    kErrEmbedToken = 1,
    kErrRopePosition = 2,
    kErrRopeBlock = 3,
    kErrAttnBlock = 4,
    kErrAttnLength = 5,
    kErrPackNonFinite = 6,
    kErrPackOverflow = 7,
    kErrGemvStage = 8,
    kErrStepBarrier = 9,
    kErrKvNonFinite = 10,
    kErrKvOverflow = 11,
    kErrMoeExpert = 12,
};
// The current device's record (allocated on first use, zero-filled).
DevError* device_error_record();
// The current device's record if one was already created, else nullptr (never allocates).
DevError* device_error_record_existing();

#ifdef __CUDACC__
__device__ __forceinline__ void record_device_error(DevError* e, int where, long long index,
                                                    long long value) {
    if (e != nullptr && atomicCAS(&e->code, 0, 1) == 0) {
        e->where = where;
        e->index = index;
        e->value = value;
    }
}
#endif

// ---------------------------------------------------------------- launch helpers
int num_sms();   // SM count of the current device (cached per device)

// Programmatic dependent launch (PDL): a kernel launched with this attribute may start while
// its predecessor in the stream is still running; it must call pdl_wait() before touching
// anything the predecessor writes. Kernels call pdl_trigger() once their own early work is
// issued so that the successor can start.
#ifdef __CUDACC__
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Ask L2 to fetch this CTA's share of [base, base + bytes): the grid splits the range into
// shares of bytes / 2^floor(log2(CTAs)) (rounded up to 16 B: between one and two even shares,
// so the first CTAs cover it all, with no integer division - this runs before the kernel's wait,
// on the path of a CTA that starts after its predecessor has ended), each thread of a CTA
// issues 16 KB pieces. A hint only (no data is returned, nothing waits): used to stream a later
// kernel's weights or constants while the current kernel runs.
__device__ __forceinline__ void l2_prefetch_share(const void* base, size_t bytes) {
    if (base == nullptr || bytes < 16) return;
    const unsigned int nblocks = gridDim.x * gridDim.y * gridDim.z;
    const size_t bid = blockIdx.x + (size_t)gridDim.x * (blockIdx.y + (size_t)gridDim.y * blockIdx.z);
    const int lg = 31 - __clz((int)nblocks);   // 2^lg <= nblocks
    const size_t share = (((bytes + ((size_t)1 << lg) - 1) >> lg) + 15) & ~(size_t)15;
    const size_t start = bid * share;
    if (start >= bytes) return;
    const size_t end = start + share < bytes ? start + share : bytes;
    const size_t nthreads = (size_t)blockDim.x * blockDim.y * blockDim.z;
    for (size_t off = start + (size_t)threadIdx.x * 16384; off < end; off += nthreads * 16384) {
        const size_t n = ((end - off) < 16384 ? (end - off) : 16384) & ~(size_t)15;
        if (n)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(static_cast<const char*>(base) + off),
                         "r"((uint32_t)n) : "memory");
    }
}
#endif

// An L2 prefetch request for the next kernel's weights (two ranges: codes and scales).
// L2 policy for data read once per step (weights, the K/V context): evicted first, so that the
// step's small reused data (activations, norm weights, tables, kernel code) stays in L2.
__device__ __forceinline__ unsigned long long l2_evict_first() {
    unsigned long long pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

struct NextWeights {
    const void* ptr[2];
    size_t bytes[2];
};

template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                   cudaStream_t s, bool pdl, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- GEMV (internal form)
enum GemvPrologue { kProX16 = 0, kProRmsF32 = 1 };
enum { kEpiArgmax = 3 };   // internal epilogue: logits (optional) + packed argmax keys

struct GemvArgs {
    const __half* scales;
    const uint8_t* quants;
    int64_t rows, cols;
    int batch;
    // input: kProX16 -> x16 [batch][cols] f16; kProRmsF32 -> xf [batch][cols] f32, normed
    // with norm_w and eps inside the kernel (RMSNorm prologue)
    int prologue;
    const __half* x16;
    const float* xf;
    const float* norm_w;
    float eps;
    int epilogue;               // QL_EPI_* or kEpiArgmax
    int y_dtype;                // QL_DTYPE_*
    void* y;
    const float* residual;
    unsigned long long* argmax_keys;   // [batch], kEpiArgmax
    const int32_t* active;      // optional, kEpiArgmax: inactive columns skip the argmax
    NextWeights next;           // optional L2 prefetch of the following kernel's weights
};
int gemv_launch(const GemvArgs& a, cudaStream_t s, bool pdl);
int gemv_prepare();   // per-device kernel attributes; call outside stream capture

// ---------------------------------------------------------------- attention (internal)
struct AttnArgs {
    const __half* q;
    const __half* k_pool;
    const __half* v_pool;
    const int32_t* block_tables;
    const int32_t* context_lens;   // if null: positions[b] + 1 (decode step form)
    const int32_t* positions;
    const int32_t* active;
    int batch, n_heads, n_kv_heads, head_dim, block_size;
    int64_t max_blocks_per_seq, num_blocks;
    float scale;
    __half* out;
    void* workspace;
    size_t workspace_bytes;
    NextWeights next;
    // fused qk-norm + RoPE + KV append (decode step); q is unused when qkv is set
    const float* qkv;
    const float* q_norm;
    const float* k_norm;
    const float* cos_t;
    const float* sin_t;
    float eps;
    int64_t max_position;
    uint8_t* kvq;                // quantised pool of the layer (keys q8_0, values q5_1) instead of
                                 // k_pool / v_pool; the fused form appends to it
    unsigned long long* trace;   // optional [CTAs][8] globaltimer stamps (CTAs with a linear index
    int trace_ctas;              // below trace_ctas): 0 start, 1 past the wait, 2 q ready,
                                 // 3 blocks done, 4 partial written / ticket taken, 5 end
};
size_t attn_workspace_bytes(int64_t batch, int n_heads, int n_kv_heads, int head_dim,
                            int block_size, int64_t max_blocks_per_seq);
int attn_launch(const AttnArgs& a, cudaStream_t s, bool pdl);
int attn_prepare();   // per-device kernel attributes; call outside stream capture

// ---------------------------------------------------------------- norm + rope (internal)
struct RopeArgs {
    const float* qkv;
    const float* q_norm;
    const float* k_norm;
    const float* cos_t;
    const float* sin_t;
    const int32_t* positions;
    const int32_t* active;
    float eps;
    int batch, n_heads, n_kv_heads, head_dim;
    __half* q_out;
    __half* k_pool;
    __half* v_pool;
    const int32_t* block_tables;
    int64_t max_blocks_per_seq;
    int block_size;
    int64_t num_blocks;
    int64_t max_position;
    NextWeights next;
};
int rope_launch(const RopeArgs& a, cudaStream_t s, bool pdl);

// ---------------------------------------------------------------- persistent decode step
// The whole step of a small batch as one cooperative kernel (one CTA per SM); see
// ql_persist.cuh. Matrices are described as the kernel streams them.
struct PMat {
    const uint8_t* stream;   // the matrix in the tile stream layout (persist_pack_streams)
    const uint8_t* quants;   // the row-major q4_0 source: codes [rows][nblk][16]
    const __half* scales;    //                            scales [rows][nblk]
    int rows, nblk;     // nblk = cols / 32, a multiple of 4
    int silu;           // rows = [gate | up]; a tile is 8 gate rows + the matching 8 up rows
    int ntile;          // 16-row tiles
    // Routed experts (stream GEMV only): a virtual matrix of nsel selected experts. Tile t of it
    // is tile t % etiles of expert sel[t / etiles] of the stream (experts are consecutive runs
    // of etiles tiles, nexp of them); rows and ntile count the virtual matrix. xsel: the
    // activation column of tile t is t / etiles (nsel columns staged), else the batch column.
    const int32_t* sel;
    int etiles, nexp, nsel, xsel;
};
// Bytes of a matrix in the tile stream layout: ntile * (nblk / 4) units of 1152 B.
size_t persist_stream_bytes(const PMat& m);
// Re-lay n matrices (quants/scales set) into `buf` (persist_stream_bytes of each, back to back)
// and set their `stream` pointers; runs on stream s.
int persist_pack_streams(PMat* mats, int n, uint8_t* buf, cudaStream_t s);
struct PLayer {
    PMat m[4];          // q|k|v, o, gate|up, down
    const float* attn_norm;
    const float* ffn_norm;
    const float* q_norm;
    const float* k_norm;
};
constexpr int kPersistMaxBatch = 2;
struct PersistParams {
    const PLayer* layers;   // device array [n_layers]
    int n_layers;
    PMat lm;
    const float* final_norm;
    const float* embed;
    int hidden, inter, vocab, nh, nkv, B, maxb, nsplit, max_nblk;
    float eps, scale_log2;
    long long num_blocks, layer_pool, max_position, out_stride;
    unsigned long long barrier_timeout_ns;
    unsigned int barrier_extra;     // arrivals every barrier waits for beyond the grid (tests: 1)
    unsigned long long* trace;      // optional [1 + barriers][grid][2] globaltimer stamps
    const int32_t* tokens;
    int32_t* positions;
    const int32_t* block_tables;
    const int32_t* active;
    int32_t* next_tokens;
    int32_t* out_tokens;
    float* logits;
    float* x;       // [B][hidden] f32 residual stream
    float* qkv;     // [B][(nh + 2 nkv) hd] f32
    __half* attn;   // [B][nh hd]
    __half* act;    // [B][inter]
    unsigned long long* keys;   // [B] packed argmax keys, zero between steps
    const float* cos_t;
    const float* sin_t;
    __half* k_pool;
    __half* v_pool;
    float* pm;      // [B][nh][nsplit] split partials of the attention
    float* pl;
    float* pacc;    // [B][nh][nsplit][hd]
    int* tickets;   // [B][nkv], zero between steps
    unsigned int* sync;   // [4], zero between steps: barrier arrivals, exits, abort flag
    DevError* err;
};
// Dynamic shared memory of the step kernel for a batch of `batch`, matrices of at most max_nblk
// blocks per row and n_layers layers.
size_t persist_smem_bytes(int batch, int max_nblk, int head_dim, int group, int n_layers);
// Sets the kernel attributes for this shape and checks that one CTA fits on every SM with a
// cooperative launch: QL_OK, or QL_EINVAL with the reason in ql_last_error().
int persist_prepare(int batch, int max_nblk, int head_dim, int group, int n_layers);
int persist_launch(const PersistParams& p, int head_dim, int group, cudaStream_t s);

// One GEMV over a matrix in the tile stream layout, batch 1 or 2, as a stand-alone kernel
// (one CTA per SM; HFMA2 products, ring of bulk copies): the launch-per-phase step's GEMV.
// epilogue: QL_EPI_NONE (f32 y), QL_EPI_ADD_RESIDUAL (f32 y += ...), QL_EPI_SILU_MUL (f16 y,
// matrix packed with silu), kEpiArgmax (f32 logits + keys). rms: xf f32 normalised with
// norm_w, else x16 f16.
struct StreamGemvArgs {
    PMat M;
    int batch, epilogue, rms;
    const float* xf;
    const __half* x16;
    const float* norm_w;
    float eps;
    void* y;
    int ld;
    unsigned long long* keys;
    const int32_t* active;
    unsigned int* sync;   // [4] zero: the abort flag of the kernel's bounded waits
    __half* xn;           // batch 3-32 with rms: [batch][cols] scratch for the RMSNorm'd input
    void* workspace;      // batch 3-32: the K windows' partial sums (batched_gemv_workspace_bytes)
    size_t workspace_bytes;
    unsigned long long* trace;   // batch 1-2, optional: [grid][8] globaltimer stamps per CTA
    NextWeights next;     // batch 1-2: constants of a later kernel, prefetched into L2
    int grid;             // batch 1-2: CTAs (0: one per SM); fewer leave SMs to the kernel before
    // batch 3-32, the RMSNorm folded into the merges (mma.sync form): a residual-epilogue GEMV
    // given ssq_out and w_next also writes xn = f16(x w_next) and the 32-row chunk sums of x^2 of
    // the new x; an RMSNorm'd GEMV given ssq_in stages xn as it is (no rms_norm_kernel) and its
    // merge applies the norm factor from those sums
    const float* ssq_in;
    float* ssq_out;
    const float* w_next;
};
// Routed experts at batch 1 (ql_moe.cu): the router + top-k kernel and the combine kernel.
struct MoeRouterArgs {
    const float* x;        // [hidden] f32 residual stream (normalised inside with norm_w)
    const float* norm_w;   // [hidden]
    const float* router;   // [num_experts][hidden] f32
    int hidden, num_experts, topk, norm_topk;
    float eps;
    float* logits;         // [num_experts] scratch
    int* ticket;           // zero between launches (re-armed by the kernel)
    int32_t* eidx;         // [topk] selected experts, by falling probability
    float* ewt;            // [topk] their weights
};
int moe_router_launch(const MoeRouterArgs& a, cudaStream_t s, bool pdl);
int moe_combine_launch(float* x, const float* y, const float* ewt, int hidden, int k, cudaStream_t s, bool pdl);

int persist_trace_words();   // trace entries per CTA and row
int stream_gemv_prepare();
int stream_gemv_launch(const StreamGemvArgs& a, cudaStream_t s, bool pdl);
// The same over batches of up to 32 (ql_batched.cu): tensor-core products, K in windows of
// 1024, every weight byte streamed once. Needs nblk / 4 < 8 or a multiple of 8.
bool batched_gemv_shape_ok(int nblk);
size_t batched_gemv_workspace_bytes(int rows, int nblk, int silu);
int batched_gemv_prepare();
int batched_gemv_launch(const StreamGemvArgs& a, cudaStream_t s, bool pdl);

}  // namespace ql
