// Per-head q/k RMSNorm + NeoX RoPE + paged KV append, one kernel.
//
// [IL] inferencelayer cuda_llm.rs CudaQwen3::step (qk_norm_rope: per-head norm when qk_norm is
// set, RoPE at the device-resident position, K and V written to the cache) and Cfg::qk_norm
// ("RMSNorm with weight 1 is NOT a no-op"); [ME] memra-engine qwen4exp_gpu.rs host_rms_norm and
// host_rope_at (split-half pairs (i, i + hd/2)); [FK] ferrum-kernels cuda_decode.rs
// attention_paged (position p goes to block_table[p / 16], slot p % 16).
//
// One CTA per (head, slot), head_dim/2 threads: thread i owns the rotation pair
// (i, i + head_dim/2). Query heads write f16 q; key heads also copy their V head into the pool.
#include <cuda_fp16.h>

#include "ql_internal.h"

namespace ql {
namespace {

struct RParams {
    const float* qkv;
    const float* q_norm;
    const float* k_norm;
    const float* cos_t;
    const float* sin_t;
    const int32_t* positions;
    const int32_t* active;
    float eps;
    int n_heads, n_kv;
    __half* q_out;
    __half* k_pool;
    __half* v_pool;
    const int32_t* block_tables;
    int maxb, bs;
    long long num_blocks;
    long long max_position;
    NextWeights next;
};

template <int HD>
__global__ void __launch_bounds__(HD / 2) norm_rope_kernel(RParams p, DevError* err) {
    constexpr int H2 = HD / 2;
    constexpr int NW = (H2 + 31) / 32;
    __shared__ float red[NW];
    const int hh = blockIdx.x, b = blockIdx.y, i = threadIdx.x;
    l2_prefetch_share(p.next.ptr[0], p.next.bytes[0]);
    l2_prefetch_share(p.next.ptr[1], p.next.bytes[1]);
    pdl_wait();
    pdl_trigger();
    if (p.active && p.active[b] == 0) return;
    const int pos = p.positions[b];
    const bool is_q = hh < p.n_heads;
    const int g = hh - p.n_heads;
    const int width = (p.n_heads + 2 * p.n_kv) * HD;
    const float* src = p.qkv + (size_t)b * width + (size_t)hh * HD;
    const float x = src[i], y = src[i + H2];
    float ss = x * x + y * y;
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (NW > 1) {
        if ((i & 31) == 0) red[i >> 5] = ss;
        __syncthreads();
        ss = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) ss += red[w];
    }
    const float r = rsqrtf(fmaf(ss, 1.0f / (float)HD, p.eps));
    const float* w = is_q ? p.q_norm : p.k_norm;
    const float xn = x * r * w[i], yn = y * r * w[i + H2];
    if (pos < 0 || pos >= p.max_position) {
        if (i == 0 && hh == 0) record_device_error(err, kErrRopePosition, b, pos);
        return;
    }
    const float c = p.cos_t[(size_t)pos * H2 + i], s = p.sin_t[(size_t)pos * H2 + i];
    const float o0 = xn * c - yn * s, o1 = xn * s + yn * c;
    if (is_q) {
        __half* q = p.q_out + ((size_t)b * p.n_heads + hh) * HD;
        q[i] = __float2half_rn(o0);
        q[i + H2] = __float2half_rn(o1);
        return;
    }
    const int lb = pos / p.bs;
    if (lb >= p.maxb) {
        if (i == 0) record_device_error(err, kErrRopePosition, b, pos);
        return;
    }
    const int phys = p.block_tables[(size_t)b * p.maxb + lb];
    if (phys < 0 || phys >= p.num_blocks) {
        if (i == 0) record_device_error(err, kErrRopeBlock, (long long)b * p.maxb + lb, phys);
        return;
    }
    const size_t off = (((size_t)phys * p.n_kv + g) * p.bs + (pos % p.bs)) * HD;
    p.k_pool[off + i] = __float2half_rn(o0);
    p.k_pool[off + i + H2] = __float2half_rn(o1);
    const float* vsrc = p.qkv + (size_t)b * width + (size_t)(p.n_heads + p.n_kv + g) * HD;
    p.v_pool[off + i] = __float2half_rn(vsrc[i]);
    p.v_pool[off + i + H2] = __float2half_rn(vsrc[i + H2]);
}

}  // namespace

int rope_launch(const RopeArgs& a, cudaStream_t s, bool pdl) {
    QL_REQUIRE(a.qkv && a.q_norm && a.k_norm && a.cos_t && a.sin_t && a.positions && a.q_out &&
                   a.k_pool && a.v_pool && a.block_tables,
               "norm_rope: null pointer");
    QL_REQUIRE(a.head_dim == 64 || a.head_dim == 128, "norm_rope: head_dim must be 64 or 128");
    QL_REQUIRE(a.n_heads > 0 && a.n_kv_heads > 0 && a.n_heads % a.n_kv_heads == 0,
               "norm_rope: bad head counts");
    QL_REQUIRE(a.batch >= 1 && a.batch <= 65535, "norm_rope: batch out of range");
    QL_REQUIRE(a.block_size == 16, "norm_rope: block_size must be 16");
    QL_REQUIRE(a.max_blocks_per_seq >= 1 && a.num_blocks >= 1 && a.max_position >= 1,
               "norm_rope: bad sizes");
    if (!device_error_record()) return set_error(QL_ECUDA, "norm_rope: no device error record");
    RParams p = {};
    p.qkv = a.qkv;
    p.q_norm = a.q_norm;
    p.k_norm = a.k_norm;
    p.cos_t = a.cos_t;
    p.sin_t = a.sin_t;
    p.positions = a.positions;
    p.active = a.active;
    p.eps = a.eps;
    p.n_heads = a.n_heads;
    p.n_kv = a.n_kv_heads;
    p.q_out = a.q_out;
    p.k_pool = a.k_pool;
    p.v_pool = a.v_pool;
    p.block_tables = a.block_tables;
    p.maxb = (int)a.max_blocks_per_seq;
    p.bs = a.block_size;
    p.num_blocks = a.num_blocks;
    p.max_position = a.max_position;
    p.next = a.next;
    dim3 grid(a.n_heads + a.n_kv_heads, a.batch);
    cudaError_t e = a.head_dim == 128
                        ? launch(norm_rope_kernel<128>, grid, dim3(64), 0, s, pdl, p, device_error_record())
                        : launch(norm_rope_kernel<64>, grid, dim3(32), 0, s, pdl, p, device_error_record());
    if (e != cudaSuccess) return cuda_error(e, "norm_rope launch");
    return QL_OK;
}

}  // namespace ql

extern "C" int ql_fused_norm_rope(const float* d_qkv, const float* d_q_norm_w, const float* d_k_norm_w,
                                  const float* d_cos, const float* d_sin, const int32_t* d_positions,
                                  const int32_t* d_active, float eps, int64_t batch, int n_heads,
                                  int n_kv_heads, int head_dim, void* d_q_out, void* d_k_pool,
                                  void* d_v_pool, const int32_t* d_block_tables,
                                  int64_t max_blocks_per_seq, int block_size, int64_t num_blocks,
                                  int64_t max_position, void* stream) {
    using namespace ql;
    if (batch < 1 || batch > 65535) return set_error(QL_EINVAL, "ql_fused_norm_rope: batch out of range");
    RopeArgs a = {};
    a.qkv = d_qkv;
    a.q_norm = d_q_norm_w;
    a.k_norm = d_k_norm_w;
    a.cos_t = d_cos;
    a.sin_t = d_sin;
    a.positions = d_positions;
    a.active = d_active;
    a.eps = eps;
    a.batch = (int)batch;
    a.n_heads = n_heads;
    a.n_kv_heads = n_kv_heads;
    a.head_dim = head_dim;
    a.q_out = static_cast<__half*>(d_q_out);
    a.k_pool = static_cast<__half*>(d_k_pool);
    a.v_pool = static_cast<__half*>(d_v_pool);
    a.block_tables = d_block_tables;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.block_size = block_size;
    a.num_blocks = num_blocks;
    a.max_position = max_position;
    return rope_launch(a, static_cast<cudaStream_t>(stream), true);
}
