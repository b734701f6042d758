// q4_0 quantiser on the GPU, bit-identical to the host codec (both use ql::q4_0_block).
// [IL] inferencelayer cuda_llm.rs: weights are quantised to q4_0 at load (up_q4) - this is the
// device-side equivalent for weights that already live in device memory.
#include "ql_f16.h"
#include "ql_internal.h"

namespace ql {
namespace {

// One thread per 32-weight block; a warp covers 32 consecutive blocks of one row range.
__global__ void __launch_bounds__(256) pack_kernel(const float* __restrict__ w, long long nblocks_total,
                                                   uint16_t* __restrict__ scales,
                                                   uint8_t* __restrict__ quants, DevError* err) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= nblocks_total) return;
    float x[32];
    const float4* src = reinterpret_cast<const float4*>(w + i * 32);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const float4 v = src[c];
        x[4 * c] = v.x;
        x[4 * c + 1] = v.y;
        x[4 * c + 2] = v.z;
        x[4 * c + 3] = v.w;
    }
    uint16_t s;
    uint8_t q[16];
    const int rc = q4_0_block(x, &s, q);
    if (rc) record_device_error(err, rc == 1 ? kErrPackNonFinite : kErrPackOverflow, i, 0);
    scales[i] = s;
    uint4 out;
    out.x = q[0] | (q[1] << 8) | (q[2] << 16) | ((uint32_t)q[3] << 24);
    out.y = q[4] | (q[5] << 8) | (q[6] << 16) | ((uint32_t)q[7] << 24);
    out.z = q[8] | (q[9] << 8) | (q[10] << 16) | ((uint32_t)q[11] << 24);
    out.w = q[12] | (q[13] << 8) | (q[14] << 16) | ((uint32_t)q[15] << 24);
    reinterpret_cast<uint4*>(quants)[i] = out;
}

}  // namespace
}  // namespace ql

extern "C" int ql_q4_0_pack_device(const float* d_w, int64_t rows, int64_t cols, void* d_scales,
                                   void* d_quants, void* stream) {
    using namespace ql;
    QL_REQUIRE(d_w && d_scales && d_quants, "ql_q4_0_pack_device: null pointer");
    QL_REQUIRE(rows > 0 && cols > 0 && cols % 32 == 0, "ql_q4_0_pack_device: need cols % 32 == 0");
    QL_REQUIRE((reinterpret_cast<uintptr_t>(d_w) & 15) == 0 && (reinterpret_cast<uintptr_t>(d_quants) & 15) == 0,
               "ql_q4_0_pack_device: weights and codes must be 16-byte aligned");
    DevError* err = device_error_record();
    if (!err) return set_error(QL_ECUDA, "ql_q4_0_pack_device: no device error record");
    const long long n = rows * (cols / 32);
    const long long grid = (n + 255) / 256;
    QL_REQUIRE(grid < (1ll << 31), "ql_q4_0_pack_device: matrix too large");
    cudaError_t e = launch(pack_kernel, dim3((unsigned)grid), dim3(256), 0, static_cast<cudaStream_t>(stream),
                           false, d_w, n, static_cast<uint16_t*>(d_scales), static_cast<uint8_t*>(d_quants), err);
    if (e != cudaSuccess) return cuda_error(e, "ql_q4_0_pack_device launch");
    return QL_OK;
}
