// Quantised KV rows on the GPU: q8_0 keys and q5_1 values, bit-identical to the host codec
// (both run the block routines of ql_kvq.h). memra-engine qwen4exp_gpu.rs keeps its device
// quantisers and host twins bit-identical in the same way.
#include "ql_internal.h"
#include "ql_kvq.h"

namespace ql {
namespace {

// One thread per 32-element block of a row; a ragged last block reads only the row's values.
template <bool Q8>
__global__ void __launch_bounds__(256) kv_quant_kernel(const float* __restrict__ x, long long rows, long long dim,
                                                       uint8_t* __restrict__ out, DevError* err) {
    const long long nblk = (dim + 31) / 32;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= rows * nblk) return;
    const long long r = i / nblk, j = i - r * nblk;
    const long long e0 = j * 32;
    const int n = (int)(dim - e0 < 32 ? dim - e0 : 32);
    float v[32];
    bool finite = true;
#pragma unroll
    for (int l = 0; l < 32; ++l) {
        v[l] = l < n ? x[r * dim + e0 + l] : 0.0f;
        finite = finite && isfinite(v[l]);
    }
    const int bb = Q8 ? kQ8Bytes : kQ5Bytes;
    uint8_t* o = out + r * nblk * bb + j * bb;
    const int rc = Q8 ? kvq_q8_block(v, n, o) : kvq_q5_block(v, n, o);
    if (!finite) record_device_error(err, kErrKvNonFinite, r, j);
    else if (rc) record_device_error(err, kErrKvOverflow, r, j);
}

// One thread per element.
template <bool Q8>
__global__ void __launch_bounds__(256) kv_dequant_kernel(const uint8_t* __restrict__ in, long long rows, long long dim,
                                                         float* __restrict__ x) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= rows * dim) return;
    const long long r = i / dim, e = i - r * dim;
    const long long nblk = (dim + 31) / 32;
    const int bb = Q8 ? kQ8Bytes : kQ5Bytes;
    const uint8_t* blk = in + r * nblk * bb + (e >> 5) * bb;
    x[i] = Q8 ? kvq_q8_value(blk, (int)(e & 31)) : kvq_q5_value(blk, (int)(e & 31));
}

template <bool Q8>
int kv_quantize_device(const char* name, const float* d_x, int64_t rows, int64_t dim, uint8_t* d_out, void* stream) {
    if (!d_x || !d_out) return set_error(QL_EINVAL, std::string(name) + ": null pointer");
    if (rows <= 0 || dim <= 0) return set_error(QL_EINVAL, std::string(name) + ": need rows > 0 and dim > 0");
    DevError* err = device_error_record();
    if (!err) return set_error(QL_ECUDA, std::string(name) + ": no device error record");
    const long long n = rows * ((dim + 31) / 32);
    const long long grid = (n + 255) / 256;
    if (grid >= (1ll << 31)) return set_error(QL_EINVAL, std::string(name) + ": too many rows");
    const cudaError_t e = launch(kv_quant_kernel<Q8>, dim3((unsigned)grid), dim3(256), 0,
                                 static_cast<cudaStream_t>(stream), false, d_x, (long long)rows, (long long)dim,
                                 d_out, err);
    return e == cudaSuccess ? QL_OK : cuda_error(e, name);
}

template <bool Q8>
int kv_dequantize_device(const char* name, const uint8_t* d_in, int64_t rows, int64_t dim, float* d_x, void* stream) {
    if (!d_in || !d_x) return set_error(QL_EINVAL, std::string(name) + ": null pointer");
    if (rows <= 0 || dim <= 0) return set_error(QL_EINVAL, std::string(name) + ": need rows > 0 and dim > 0");
    const long long n = rows * dim;
    const long long grid = (n + 255) / 256;
    if (grid >= (1ll << 31)) return set_error(QL_EINVAL, std::string(name) + ": too many rows");
    const cudaError_t e = launch(kv_dequant_kernel<Q8>, dim3((unsigned)grid), dim3(256), 0,
                                 static_cast<cudaStream_t>(stream), false, d_in, (long long)rows, (long long)dim, d_x);
    return e == cudaSuccess ? QL_OK : cuda_error(e, name);
}

}  // namespace
}  // namespace ql

extern "C" int ql_kv_quantize_q8_0_device(const float* d_x, int64_t rows, int64_t dim, uint8_t* d_out,
                                          void* stream) {
    return ql::kv_quantize_device<true>("ql_kv_quantize_q8_0_device", d_x, rows, dim, d_out, stream);
}

extern "C" int ql_kv_quantize_q5_1_device(const float* d_x, int64_t rows, int64_t dim, uint8_t* d_out,
                                          void* stream) {
    return ql::kv_quantize_device<false>("ql_kv_quantize_q5_1_device", d_x, rows, dim, d_out, stream);
}

extern "C" int ql_kv_dequantize_q8_0_device(const uint8_t* d_in, int64_t rows, int64_t dim, float* d_x,
                                            void* stream) {
    return ql::kv_dequantize_device<true>("ql_kv_dequantize_q8_0_device", d_in, rows, dim, d_x, stream);
}

extern "C" int ql_kv_dequantize_q5_1_device(const uint8_t* d_in, int64_t rows, int64_t dim, float* d_x,
                                            void* stream) {
    return ql::kv_dequantize_device<false>("ql_kv_dequantize_q5_1_device", d_in, rows, dim, d_x, stream);
}

// ---------------------------------------------------------------- the quantised attention pool
#include "ql_kvq_rec.cuh"

namespace ql {
namespace {

// One warp per (row i, kv head g): key row i and value row i of kv head g quantised into slot
// slots[i] % 16 of the record of physical block slots[i] / 16 (the warp-level routines of the
// attention's fused append, so a row written here reads back exactly as one appended there).
template <int HD>
__global__ void __launch_bounds__(256) kvq_write_kernel(const float* __restrict__ k, const float* __restrict__ v,
                                                        const long long* __restrict__ slots, long long n, int n_kv,
                                                        uint8_t* __restrict__ pool, long long num_blocks,
                                                        DevError* err) {
    const long long wi = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wi >= n * n_kv) return;   // uniform per warp
    const long long i = wi / n_kv;
    const int g = (int)(wi - i * n_kv);
    const long long slot = slots[i];
    const long long blk = slot >> 4;
    if (slot < 0 || blk >= num_blocks) {
        if (lane == 0 && g == 0) record_device_error(err, kErrAttnBlock, i, slot);
        return;
    }
    const float* kr = k + (size_t)wi * HD;
    const float* vr = v + (size_t)wi * HD;
    float xk[HD / 32], xv[HD / 32];
    bool finite = true;
#pragma unroll
    for (int c = 0; c < HD / 32; ++c) {
        xk[c] = kr[32 * c + lane];
        xv[c] = vr[32 * c + lane];
        finite = finite && isfinite(xk[c]) && isfinite(xv[c]);
    }
    finite = __all_sync(0xffffffffu, finite);
    uint8_t* rec = pool + ((size_t)blk * n_kv + g) * Kvq<HD>::BYTES;
    const int s = (int)(slot & 15);
    const bool okk = kvq_put_k_row<HD>(xk, rec, s, lane, nullptr);
    const bool okv = kvq_put_v_row<HD>(xv, rec, s, lane, nullptr);
    if (lane == 0 && !finite) record_device_error(err, kErrKvNonFinite, i, g);
    else if (lane == 0 && !(okk && okv)) record_device_error(err, kErrKvOverflow, i, g);
}

}  // namespace
}  // namespace ql

extern "C" int64_t ql_kvq_record_bytes(int head_dim) {
    return (head_dim == 64 || head_dim == 128) ? (int64_t)29 * head_dim : 0;
}

extern "C" int ql_kvq_write(const float* d_k, const float* d_v, const int64_t* d_slots, int64_t n, int n_kv_heads,
                            int head_dim, void* d_pool, int64_t num_blocks, void* stream) {
    using namespace ql;
    QL_REQUIRE(d_k && d_v && d_slots && d_pool, "ql_kvq_write: null pointer");
    QL_REQUIRE(head_dim == 64 || head_dim == 128, "ql_kvq_write: head_dim must be 64 or 128");
    QL_REQUIRE(n > 0 && n_kv_heads > 0 && num_blocks > 0, "ql_kvq_write: need n, n_kv_heads and num_blocks > 0");
    QL_REQUIRE((reinterpret_cast<uintptr_t>(d_pool) & 15) == 0, "ql_kvq_write: the pool must be 16-byte aligned");
    DevError* err = device_error_record();
    if (!err) return set_error(QL_ECUDA, "ql_kvq_write: no device error record");
    const long long warps = n * n_kv_heads;
    const long long grid = (warps * 32 + 255) / 256;
    QL_REQUIRE(grid < (1ll << 31), "ql_kvq_write: too many rows");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const long long* sl = reinterpret_cast<const long long*>(d_slots);
    uint8_t* pool = static_cast<uint8_t*>(d_pool);
    const cudaError_t e =
        head_dim == 128 ? launch(kvq_write_kernel<128>, dim3((unsigned)grid), dim3(256), 0, s, false, d_k, d_v, sl,
                                 (long long)n, n_kv_heads, pool, (long long)num_blocks, err)
                        : launch(kvq_write_kernel<64>, dim3((unsigned)grid), dim3(256), 0, s, false, d_k, d_v, sl,
                                 (long long)n, n_kv_heads, pool, (long long)num_blocks, err);
    return e == cudaSuccess ? QL_OK : cuda_error(e, "ql_kvq_write");
}
