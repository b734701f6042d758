// q4_0 GEMV on the CUDA cores: y[b][r] = sum_k (q[r][k] - 8) * d[r][k/32] * x[b][k].
//
// [IL] inferencelayer cuda_llm.rs, CudaQwen3::gemv / Q4Dev (the q4_0 format and the
// one-GEMV-per-projection dataflow, fused q|k|v and gate|up rows).
//
// Design (GB300): the step is HBM-bound weight streaming, so the kernel is built around the
// instruction budget per weight rather than around the tensor cores:
//  * each lane streams whole 32-weight blocks (16 code bytes, one 16-byte load per row) of R
//    rows at once; a warp covers 32 consecutive blocks of a row, so every load instruction
//    of a warp reads 512 contiguous bytes per row;
//  * the activation vector is staged once per CTA in shared memory as f16, permuted so that
//    one 16-byte shared load yields exactly the four f16 pairs that match the four code pairs
//    a 32-bit code word expands to, and swizzled so that the 8 lanes of a quarter-warp hit 8
//    different bank groups; each staged chunk is reused by the R rows of a task;
//  * a 32-bit code word expands to four f16x2 values with one shift and four LOP3s: a nibble
//    OR'ed into the mantissa of 1024.0h gives 1024 + q exactly; the high nibbles land 4 bits
//    up (1024 + 16 q) and their activations are staged pre-divided by 16 (exact);
//    subtracting 1032 (resp. 1152) gives (q - 8) (resp. 16 (q - 8)) exactly;
//  * the 32 products of a block accumulate in f16x2 (16 terms per half), and each block's sum
//    is scaled by d and accumulated in f32;
//  * the CTA's rows are contiguous, so its first bytes are prefetched into L2 before the
//    kernel waits on its predecessor (programmatic dependent launch).
// Fused prologue: RMSNorm of an f32 residual stream (x / sqrt(mean(x^2) + eps) * w, [ME]
// host_rms_norm) into the staged f16 activations. Fused epilogues: residual add, SiLU * up
// (gate | up rows), and greedy argmax over the rows (lm_head).
#include <cuda_fp16.h>

#include <mutex>
#include <set>

#include "ql_internal.h"

namespace ql {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr size_t kMaxStageBytes = 100 * 1024;   // staged activations per CTA

__device__ __forceinline__ int xslot(int j, int i) { return (j << 2) + (i ^ ((j >> 1) & 3)); }

__device__ __forceinline__ __half2 h2(uint32_t u) {
    __half2 h;
    *reinterpret_cast<uint32_t*>(&h) = u;
    return h;
}
__device__ __forceinline__ uint32_t u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

// Order-preserving key: larger logit -> larger key; among equal logits the lower row wins.
__device__ __forceinline__ unsigned long long argmax_key(float v, int row) {
    uint32_t b = __float_as_uint(v);
    b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return ((unsigned long long)b << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)row);
}

struct KParams {
    const __half* scales;
    const uint8_t* quants;
    int rows;          // weight rows
    int nblk;          // cols / 32
    int batch;         // columns handled by this launch (<= NB)
    int prologue;
    const __half* x16; // [batch][cols]
    const float* xf;   // [batch][cols]
    const float* norm_w;
    float eps;
    int epilogue;
    int y_dtype;
    void* y;
    int y_ld;          // row stride of y / residual (elements)
    const float* residual;
    unsigned long long* keys;
    const int32_t* active;
    int ntasks;
    int tasks_per_cta;
};

// Stage the activation columns into shared memory in the permuted, swizzled chunk layout.
template <int NB>
__device__ void stage_x(const KParams& p, uint4* xs, float* red) {
    const int cols = p.nblk * 32;
    const int tid = threadIdx.x;
    float rs[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) rs[b] = 1.0f;
    if (p.prologue == kProRmsF32) {
        float ss[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            ss[b] = 0.f;
            if (b < p.batch) {
                const float4* xb = reinterpret_cast<const float4*>(p.xf + (size_t)b * cols);
                for (int k = tid; k < cols / 4; k += kThreads) {
                    const float4 v = xb[k];
                    ss[b] += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
                }
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) ss[b] += __shfl_xor_sync(0xffffffffu, ss[b], o);
        }
        const int warp = tid >> 5, lane = tid & 31;
        if (lane == 0) {
#pragma unroll
            for (int b = 0; b < NB; ++b) red[warp * NB + b] = ss[b];
        }
        __syncthreads();
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            float t = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) t += red[w * NB + b];
            rs[b] = 1.0f / sqrtf(t / (float)cols + p.eps);
        }
    }
    const int nchunk = p.nblk * 4;
    for (int c = tid; c < NB * nchunk; c += kThreads) {
        const int b = c / nchunk;
        const int rem = c - b * nchunk;
        const int j = rem >> 2, i = rem & 3;
        float lo[4], hi[4];   // x[32j + 4i + 0..3], x[32j + 16 + 4i + 0..3]
        if (b < p.batch) {
            const size_t base = (size_t)b * cols + 32 * j + 4 * i;
            if (p.prologue == kProRmsF32) {
                const float4 a = *reinterpret_cast<const float4*>(p.xf + base);
                const float4 h = *reinterpret_cast<const float4*>(p.xf + base + 16);
                const float4 wa = *reinterpret_cast<const float4*>(p.norm_w + 32 * j + 4 * i);
                const float4 wh = *reinterpret_cast<const float4*>(p.norm_w + 32 * j + 16 + 4 * i);
                float rr = rs[0];
#pragma unroll
                for (int bb = 0; bb < NB; ++bb)
                    if (bb == b) rr = rs[bb];
                // RMSNorm output rounded to f16 (the GEMV's activation precision)
                lo[0] = __half2float(__float2half_rn(a.x * rr * wa.x));
                lo[1] = __half2float(__float2half_rn(a.y * rr * wa.y));
                lo[2] = __half2float(__float2half_rn(a.z * rr * wa.z));
                lo[3] = __half2float(__float2half_rn(a.w * rr * wa.w));
                hi[0] = __half2float(__float2half_rn(h.x * rr * wh.x));
                hi[1] = __half2float(__float2half_rn(h.y * rr * wh.y));
                hi[2] = __half2float(__float2half_rn(h.z * rr * wh.z));
                hi[3] = __half2float(__float2half_rn(h.w * rr * wh.w));
            } else {
                const uint2 a = *reinterpret_cast<const uint2*>(p.x16 + base);
                const uint2 h = *reinterpret_cast<const uint2*>(p.x16 + base + 16);
                const float2 a0 = __half22float2(h2(a.x)), a1 = __half22float2(h2(a.y));
                const float2 h0 = __half22float2(h2(h.x)), h1 = __half22float2(h2(h.y));
                lo[0] = a0.x; lo[1] = a0.y; lo[2] = a1.x; lo[3] = a1.y;
                hi[0] = h0.x; hi[1] = h0.y; hi[2] = h1.x; hi[3] = h1.y;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) lo[e] = hi[e] = 0.f;
        }
        uint4 v;
        v.x = u32(__floats2half2_rn(lo[0], lo[2]));
        v.y = u32(__floats2half2_rn(lo[1], lo[3]));
        v.z = u32(__floats2half2_rn(hi[0] * 0.0625f, hi[2] * 0.0625f));
        v.w = u32(__floats2half2_rn(hi[1] * 0.0625f, hi[3] * 0.0625f));
        xs[b * nchunk + xslot(j, i)] = v;
    }
}

// Reduce a task's per-lane partial sums over the warp and apply the epilogue.
template <int NB, int R>
__device__ __forceinline__ void epilogue_task(const KParams& p, int t, float (&acc)[R][NB], int lane,
                                              bool silu_mul, int half_rows,
                                              unsigned long long (&best)[NB]) {
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int b = 0; b < NB; ++b)
#pragma unroll
            for (int o = 16; o; o >>= 1) acc[r][b] += __shfl_xor_sync(0xffffffffu, acc[r][b], o);
    int row[R];
    bool ok[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (silu_mul) {
            const int i = t * (R / 2) + (r % (R / 2));
            ok[r] = i < half_rows;
            row[r] = (r < R / 2) ? i : half_rows + i;
        } else {
            row[r] = t * R + r;
            ok[r] = row[r] < p.rows;
        }
    }
    // lane l writes output number l (R * NB <= 32)
    if (silu_mul) {
#pragma unroll
        for (int r = 0; r < R / 2; ++r)
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (lane == r * NB + b && ok[r] && b < p.batch) {
                    const float v = silu(acc[r][b]) * acc[r + R / 2][b];
                    const size_t o = (size_t)b * p.y_ld + row[r];
                    if (p.y_dtype == QL_DTYPE_F16)
                        reinterpret_cast<__half*>(p.y)[o] = __float2half_rn(v);
                    else
                        reinterpret_cast<float*>(p.y)[o] = v;
                }
            }
    } else if (p.epilogue == kEpiArgmax) {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (ok[r] && b < p.batch) {
                    const unsigned long long k = argmax_key(acc[r][b], row[r]);
                    best[b] = k > best[b] ? k : best[b];
                    if (p.y && lane == r * NB + b)
                        reinterpret_cast<float*>(p.y)[(size_t)b * p.y_ld + row[r]] = acc[r][b];
                }
            }
    } else {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (lane == r * NB + b && ok[r] && b < p.batch) {
                    const size_t o = (size_t)b * p.y_ld + row[r];
                    float v = acc[r][b];
                    if (p.epilogue == QL_EPI_ADD_RESIDUAL) v += p.residual[o];
                    if (p.y_dtype == QL_DTYPE_F16)
                        reinterpret_cast<__half*>(p.y)[o] = __float2half_rn(v);
                    else
                        reinterpret_cast<float*>(p.y)[o] = v;
                }
            }
    }
}

template <int NB, int R>
__global__ void __launch_bounds__(kThreads, 2) gemv_q4_0_kernel(KParams p, DevError* err) {
    extern __shared__ uint4 xs[];
    __shared__ float red[kWarps * 8];
    __shared__ unsigned long long kred[kWarps * 8];
    (void)err;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool silu_mul = (p.epilogue == QL_EPI_SILU_MUL);
    const int half_rows = p.rows >> 1;
    const int t0 = blockIdx.x * p.tasks_per_cta;
    const int t1 = min(p.ntasks, t0 + p.tasks_per_cta);

    // Weights do not depend on the previous kernel: warm L2 with the start of this CTA's rows
    // while the predecessor finishes.
    if (threadIdx.x == 0 && t0 < t1) {
        const size_t row_bytes = (size_t)p.nblk * 16;
        const int nr = silu_mul ? (t1 - t0) * (R / 2) : (t1 - t0) * R;
        const int r0 = silu_mul ? t0 * (R / 2) : t0 * R;
        const int limit = silu_mul ? half_rows : p.rows;   // rows of one range
        size_t bytes = row_bytes * (size_t)min(nr, limit - r0);
        bytes = bytes > 65536 ? 65536 : bytes;
        const uint8_t* a0 = p.quants + (size_t)r0 * row_bytes;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a0), "r"((uint32_t)bytes)
                     : "memory");
        if (silu_mul) {
            const uint8_t* a1 = p.quants + (size_t)(half_rows + r0) * row_bytes;
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a1),
                         "r"((uint32_t)bytes)
                         : "memory");
        }
    }
    pdl_wait();
    stage_x<NB>(p, xs, red);
    __syncthreads();
    pdl_trigger();

    const int nchunk = p.nblk * 4;
    const __half2 k1032 = __float2half2_rn(1032.0f);
    const __half2 k1152 = __float2half2_rn(1152.0f);
    unsigned long long best[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) best[b] = 0ull;

    // Each warp walks a flat sequence of (task, 32-block step) iterations. The loads of the
    // next D iterations are always in flight, across task boundaries, so every lane keeps
    // D * R * 16 bytes of weight codes outstanding.
    constexpr int D = NB >= 4 ? 2 : (NB == 2 && R == 4) ? 3 : 4;
    const int njit = (p.nblk + 31) >> 5;
    const int my_tasks = (t1 - t0 > warp) ? (t1 - t0 - warp + kWarps - 1) / kWarps : 0;
    const int total = my_tasks * njit;

    auto row_of = [&](int t, int r, bool& ok) -> int {
        if (silu_mul) {
            const int i = t * (R / 2) + (r % (R / 2));
            ok = i < half_rows;
            return ok ? ((r < R / 2) ? i : half_rows + i) : 0;
        }
        const int rr = t * R + r;
        ok = rr < p.rows;
        return ok ? rr : 0;
    };
    // Load cursor: runs D iterations ahead of the compute cursor; row pointers are set once per
    // task and advanced by 32 blocks per iteration (no per-iteration index arithmetic).
    const uint4* q4 = reinterpret_cast<const uint4*>(p.quants);
    int ltask = t0 + warp, ljs = 0;
    int loff[R];     // element index row * nblk + j of the next load, per row (< 2^31)
    bool lok[R];
    auto set_rows = [&](int t) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            bool ok;
            const int row = row_of(t, r, ok);
            lok[r] = ok;
            loff[r] = row * p.nblk + lane;
        }
    };
    set_rows(ltask);
    auto issue = [&](uint4 (&qv)[R], __half (&sv)[R]) {
        const bool jok = (ljs << 5) + lane < p.nblk;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (lok[r] && jok) {
                qv[r] = __ldg(q4 + loff[r]);
                sv[r] = p.scales[loff[r]];
            } else {
                qv[r] = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
                sv[r] = __float2half(0.f);
            }
            loff[r] += 32;
        }
        if (++ljs == njit) {
            ljs = 0;
            ltask += kWarps;
            set_rows(ltask);
        }
    };

    uint4 ring[D][R];
    __half sring[D][R];
#pragma unroll
    for (int u = 0; u < D; ++u)
        if (u < total) issue(ring[u], sring[u]);

    float acc[R][NB];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int b = 0; b < NB; ++b) acc[r][b] = 0.f;

    int cjs = 0, ctask = t0 + warp;
    for (int it0 = 0; it0 < total; it0 += D) {
#pragma unroll
        for (int u = 0; u < D; ++u) {
            const int it = it0 + u;
            if (it < total) {
                const int j = (cjs << 5) + lane;
                if (j < p.nblk) {
                    const int xb = j << 2, sw = (j >> 1) & 3;
                    __half2 a[R][NB];
#pragma unroll
                    for (int r = 0; r < R; ++r)
#pragma unroll
                        for (int b = 0; b < NB; ++b) a[r][b] = __float2half2_rn(0.f);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint4 X[NB];
#pragma unroll
                        for (int b = 0; b < NB; ++b) X[b] = xs[b * nchunk + xb + (i ^ sw)];
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            const uint4 qv = ring[u][r];
                            const uint32_t w = (i == 0) ? qv.x : (i == 1) ? qv.y : (i == 2) ? qv.z : qv.w;
                            const uint32_t s8 = w >> 8;
                            const __half2 lo0 = __hsub2(h2((w & 0x000F000Fu) | 0x64006400u), k1032);
                            const __half2 hi0 = __hsub2(h2((w & 0x00F000F0u) | 0x64006400u), k1152);
                            const __half2 lo1 = __hsub2(h2((s8 & 0x000F000Fu) | 0x64006400u), k1032);
                            const __half2 hi1 = __hsub2(h2((s8 & 0x00F000F0u) | 0x64006400u), k1152);
#pragma unroll
                            for (int b = 0; b < NB; ++b) {
                                a[r][b] = __hfma2(lo0, h2(X[b].x), a[r][b]);
                                a[r][b] = __hfma2(lo1, h2(X[b].y), a[r][b]);
                                a[r][b] = __hfma2(hi0, h2(X[b].z), a[r][b]);
                                a[r][b] = __hfma2(hi1, h2(X[b].w), a[r][b]);
                            }
                        }
                    }
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const float d = __half2float(sring[u][r]);
#pragma unroll
                        for (int b = 0; b < NB; ++b) {
                            const float2 f = __half22float2(a[r][b]);
                            acc[r][b] = fmaf(d, f.x + f.y, acc[r][b]);
                        }
                    }
                }
                if (it + D < total) issue(ring[u], sring[u]);
                if (++cjs == njit) {
                    epilogue_task<NB, R>(p, ctask, acc, lane, silu_mul, half_rows, best);
#pragma unroll
                    for (int r = 0; r < R; ++r)
#pragma unroll
                        for (int b = 0; b < NB; ++b) acc[r][b] = 0.f;
                    cjs = 0;
                    ctask += kWarps;
                }
            }
        }
    }
    if (p.epilogue == kEpiArgmax) {
        // every lane holds the same per-warp maxima; reduce across the CTA, one atomic each
        if (lane == 0) {
#pragma unroll
            for (int b = 0; b < NB; ++b) kred[warp * NB + b] = best[b];
        }
        __syncthreads();
        if (threadIdx.x < NB && (int)threadIdx.x < p.batch) {
            const int b = threadIdx.x;
            unsigned long long m = 0ull;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) m = kred[w * NB + b] > m ? kred[w * NB + b] : m;
            const bool act = p.active == nullptr || p.active[b] != 0;
            if (m && act) atomicMax(p.keys + b, m);
        }
    }
}

template <int NB, int R>
cudaError_t launch_nb(const KParams& p0, int grid, size_t smem, cudaStream_t s, bool pdl) {
    return launch(gemv_q4_0_kernel<NB, R>, dim3(grid), dim3(kThreads), smem, s, pdl, p0,
                  device_error_record());
}

template <int NB, int R>
cudaError_t allow_smem() {
    return cudaFuncSetAttribute(gemv_q4_0_kernel<NB, R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kMaxStageBytes);
}

}  // namespace

// Kernel attributes are set once per device, outside any stream capture.
int gemv_prepare() {
    static std::mutex mu;
    static std::set<int> done;
    int dev = 0;
    QL_TRY_CUDA(cudaGetDevice(&dev));
    std::lock_guard<std::mutex> lk(mu);
    if (done.count(dev)) return QL_OK;
    cudaError_t e = allow_smem<1, 4>();
    if (e == cudaSuccess) e = allow_smem<2, 4>();
    if (e == cudaSuccess) e = allow_smem<1, 2>();
    if (e == cudaSuccess) e = allow_smem<2, 2>();
    if (e == cudaSuccess) e = allow_smem<4, 2>();
    if (e == cudaSuccess) e = allow_smem<8, 2>();
    if (e != cudaSuccess) return cuda_error(e, "gemv: cudaFuncSetAttribute");
    done.insert(dev);
    return QL_OK;
}

int gemv_launch(const GemvArgs& a, cudaStream_t s, bool pdl) {
    QL_REQUIRE(a.scales && a.quants && a.y, "gemv: null pointer");
    QL_REQUIRE(a.rows > 0 && a.cols > 0 && a.cols % 32 == 0, "gemv: need rows > 0, cols % 32 == 0");
    QL_REQUIRE(a.rows < (1ll << 31) && a.cols < (1ll << 24) && a.rows * (a.cols / 32) < (1ll << 31),
               "gemv: matrix too large");
    QL_REQUIRE(a.batch >= 1 && a.batch <= 64, "gemv: batch must be in [1, 64]");
    QL_REQUIRE(a.prologue == kProX16 ? a.x16 != nullptr : (a.xf && a.norm_w), "gemv: null input");
    QL_REQUIRE(a.epilogue != QL_EPI_SILU_MUL || a.rows % 2 == 0, "gemv: silu_mul needs even rows");
    QL_REQUIRE(a.epilogue != QL_EPI_ADD_RESIDUAL || (a.residual && a.y_dtype == QL_DTYPE_F32),
               "gemv: residual epilogue needs an f32 residual and f32 output");
    QL_REQUIRE(a.epilogue != kEpiArgmax || a.argmax_keys, "gemv: argmax needs key buffer");
    QL_REQUIRE(a.y_dtype == QL_DTYPE_F32 || a.y_dtype == QL_DTYPE_F16, "gemv: bad y dtype");
    QL_REQUIRE(a.epilogue != kEpiArgmax || a.y_dtype == QL_DTYPE_F32, "gemv: argmax logits are f32");
    if (!device_error_record()) return set_error(QL_ECUDA, "gemv: no device error record");
    if (int rc = gemv_prepare()) return rc;

    const int nblk = (int)(a.cols / 32);
    const size_t col_bytes = (size_t)nblk * 64;
    int nb_max = (int)(kMaxStageBytes / col_bytes);
    QL_REQUIRE(nb_max >= 1, "gemv: cols too large for the staged activation");
    nb_max = nb_max >= 8 ? 8 : nb_max >= 4 ? 4 : nb_max >= 2 ? 2 : 1;
    const int out_ld = (int)(a.epilogue == QL_EPI_SILU_MUL ? a.rows / 2 : a.rows);
    const int sms = num_sms();

    for (int b0 = 0; b0 < a.batch; b0 += nb_max) {
        const int nb = a.batch - b0 < nb_max ? a.batch - b0 : nb_max;
        const int NB = nb <= 1 ? 1 : nb <= 2 ? 2 : nb <= 4 ? 4 : 8;
        KParams p = {};
        p.scales = a.scales;
        p.quants = a.quants;
        p.rows = (int)a.rows;
        p.nblk = nblk;
        p.batch = nb;
        p.prologue = a.prologue;
        p.x16 = a.x16 ? a.x16 + (size_t)b0 * a.cols : nullptr;
        p.xf = a.xf ? a.xf + (size_t)b0 * a.cols : nullptr;
        p.norm_w = a.norm_w;
        p.eps = a.eps;
        p.epilogue = a.epilogue;
        p.y_dtype = a.y_dtype;
        const size_t esz = a.y_dtype == QL_DTYPE_F16 ? 2 : 4;
        p.y = a.y ? (void*)((char*)a.y + (size_t)b0 * out_ld * esz) : nullptr;
        p.y_ld = out_ld;
        p.residual = a.residual ? a.residual + (size_t)b0 * out_ld : nullptr;
        p.keys = a.argmax_keys ? a.argmax_keys + b0 : nullptr;
        p.active = a.active ? a.active + b0 : nullptr;
        // rows per warp task: 4 when there is enough work to fill the GPU, else 2
        const int eff_rows = (int)(a.epilogue == QL_EPI_SILU_MUL ? a.rows / 2 : a.rows);
        const int per_task_4 = a.epilogue == QL_EPI_SILU_MUL ? 2 : 4;
        const bool use4 = NB <= 2 && (eff_rows + per_task_4 - 1) / per_task_4 >= 2 * kWarps * sms;
        const int R = use4 ? 4 : 2;
        const int per_task = a.epilogue == QL_EPI_SILU_MUL ? R / 2 : R;
        p.ntasks = (eff_rows + per_task - 1) / per_task;
        int grid = (p.ntasks + kWarps - 1) / kWarps;
        if (grid > 2 * sms) grid = 2 * sms;
        p.tasks_per_cta = (p.ntasks + grid - 1) / grid;
        grid = (p.ntasks + p.tasks_per_cta - 1) / p.tasks_per_cta;
        const size_t smem = (size_t)NB * col_bytes;
        cudaError_t e;
        if (R == 4) {
            e = NB == 1 ? launch_nb<1, 4>(p, grid, smem, s, pdl) : launch_nb<2, 4>(p, grid, smem, s, pdl);
        } else {
            switch (NB) {
                case 1: e = launch_nb<1, 2>(p, grid, smem, s, pdl); break;
                case 2: e = launch_nb<2, 2>(p, grid, smem, s, pdl); break;
                case 4: e = launch_nb<4, 2>(p, grid, smem, s, pdl); break;
                default: e = launch_nb<8, 2>(p, grid, smem, s, pdl); break;
            }
        }
        if (e != cudaSuccess) return cuda_error(e, "gemv launch");
    }
    return QL_OK;
}

}  // namespace ql

extern "C" int ql_gemv_q4_0(const void* d_scales, const void* d_quants, int64_t rows, int64_t cols,
                            const void* d_x, int64_t batch, void* d_y, int y_dtype, int epilogue,
                            const float* d_residual, void* stream) {
    using namespace ql;
    if (epilogue != QL_EPI_NONE && epilogue != QL_EPI_ADD_RESIDUAL && epilogue != QL_EPI_SILU_MUL)
        return set_error(QL_EINVAL, "ql_gemv_q4_0: unknown epilogue");
    GemvArgs a = {};
    a.scales = static_cast<const __half*>(d_scales);
    a.quants = static_cast<const uint8_t*>(d_quants);
    a.rows = rows;
    a.cols = cols;
    if (batch < 1 || batch > 64) return set_error(QL_EINVAL, "ql_gemv_q4_0: batch must be in [1, 64]");
    a.batch = (int)batch;
    a.prologue = kProX16;
    a.x16 = static_cast<const __half*>(d_x);
    a.epilogue = epilogue;
    a.y_dtype = y_dtype;
    a.y = d_y;
    a.residual = d_residual;
    return gemv_launch(a, static_cast<cudaStream_t>(stream), true);
}
