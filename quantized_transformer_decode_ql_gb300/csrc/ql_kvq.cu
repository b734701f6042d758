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
