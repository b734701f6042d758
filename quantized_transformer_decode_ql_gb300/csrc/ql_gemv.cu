// q4_0 GEMV for batch <= 8 per pass: y[b][r] = sum_k (q[r][k] - 8) * d[r][k/32] * x[b][k].
//
// [IL] inferencelayer cuda_llm.rs, CudaQwen3::gemv / Q4Dev (the q4_0 format and the
// one-GEMV-per-projection dataflow, fused q|k|v and gate|up rows).
//
// Design (GB300). The step is HBM-bound weight streaming, and at 18 bytes per 32 weights the
// GPU must retire ~1.2e13 weights/s: the instruction mix per weight decides whether the HBM
// bound is reachable. Measured with ncu on an f16x2 CUDA-core variant of this kernel, the f16
// FMA/add pipe (64 lanes/clk/SM on this part, half the f32 rate) and the integer pipe were the
// limit at ~45% of HBM. This kernel therefore feeds the dot products to mma.sync (m16n8k16,
// f16 in, f32 accumulate) and keeps the CUDA cores for the nibble expansion only:
//  * a warp owns a 16-row tile (SiLU*up: 8 gate rows + the matching 8 up rows) and walks the
//    32-weight blocks of one K segment; lane (g, t) = (lane / 4, lane % 4) loads 32-bit code
//    word t of block j for rows g and g + 8, so the 4 lanes of a row read the block's 16 bytes;
//    code loads run kD blocks ahead (a register ring);
//  * one shift and four LOP3 turn a code word into four f16 pairs 1024 + q (low nibbles) and
//    1024 + 16 q (high nibbles), exactly; each pair lands in the A-fragment slots of the k
//    values it holds (any k permutation is allowed as long as B uses the same one);
//  * the activation columns are staged once per CTA in shared memory, permuted so that one
//    16-byte load gives the B fragments of both MMAs of a block, high-nibble activations
//    pre-divided by 16 (exact);
//  * the offsets are folded into the accumulator: the MMA computes sum (1024 + q) x, and the
//    accumulator starts at -(1032 sum_lo x + 1152 sum_hi x/16) per (block, column), computed
//    once per CTA from the staged values, so no f16 subtraction is executed per weight;
//  * per block, the f32 result is scaled by the row's f16 scale with one FFMA per output.
// Small matrices split K over up to 8 warps of a CTA and reduce in shared memory, so that every
// shape fills the GPU. The CTA's first codes are prefetched into L2 before the kernel waits on
// its predecessor (programmatic dependent launch).
// Fused prologue: RMSNorm of an f32 residual stream ([ME] host_rms_norm) into the staged f16
// activations. Fused epilogues: residual add, SiLU * up, greedy argmax over the rows (lm_head).
#include <cuda_fp16.h>

#include <mutex>
#include <set>

#include "ql_internal.h"

namespace ql {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kD = 8;                            // blocks of code loads in flight per lane
constexpr size_t kMaxStageBytes = 100 * 1024;    // dynamic shared memory per CTA

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

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

struct KParams {
    const __half* scales;
    const uint8_t* quants;
    int rows;          // weight rows
    int nblk;          // cols / 32
    int batch;         // columns of this launch (<= 8)
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
    int ntile;         // 16-row tiles (SiLU*up: 8 gate + 8 up rows)
    int S;             // K segments per tile (1, 2, 4 or 8 warps)
    int seg_blocks;    // blocks per K segment
    int cstride;       // uint4 units between staged columns
};

// Stage the activations: per column, per block j, 4 chunks of 16 bytes (chunk t serves lane
// t of the MMA), plus the accumulator start value of each (block, column).
__device__ void stage_x(const KParams& p, uint4* xs, float* bias, float* red) {
    const int cols = p.nblk * 32;
    const int tid = threadIdx.x;
    float rs[8];
#pragma unroll
    for (int b = 0; b < 8; ++b) rs[b] = 1.0f;
    if (p.prologue == kProRmsF32) {
        const int warp = tid >> 5, lane = tid & 31;
        for (int b = 0; b < p.batch; ++b) {
            float ss = 0.f;
            const float4* xb = reinterpret_cast<const float4*>(p.xf + (size_t)b * cols);
            for (int k = tid; k < cols / 4; k += kThreads) {
                const float4 v = xb[k];
                ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            if (lane == 0) red[warp * 8 + b] = ss;
        }
        __syncthreads();
        for (int b = 0; b < p.batch; ++b) {
            float t = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) t += red[w * 8 + b];
            const float r = 1.0f / sqrtf(t / (float)cols + p.eps);
#pragma unroll
            for (int bb = 0; bb < 8; ++bb)
                if (bb == b) rs[bb] = r;
        }
        __syncthreads();   // red is reused later
    }
    for (int item = tid; item < 8 * p.nblk; item += kThreads) {
        const int b = item / p.nblk, j = item - b * p.nblk;
        if (b >= p.batch) {
            bias[j * 8 + b] = 0.f;
            continue;
        }
        float v[32];
        const size_t base = (size_t)b * cols + 32 * j;
        if (p.prologue == kProRmsF32) {
            float rr = rs[0];
#pragma unroll
            for (int bb = 1; bb < 8; ++bb)
                if (bb == b) rr = rs[bb];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 a = *reinterpret_cast<const float4*>(p.xf + base + 4 * c);
                const float4 w = *reinterpret_cast<const float4*>(p.norm_w + 32 * j + 4 * c);
                v[4 * c + 0] = __half2float(__float2half_rn(a.x * rr * w.x));
                v[4 * c + 1] = __half2float(__float2half_rn(a.y * rr * w.y));
                v[4 * c + 2] = __half2float(__float2half_rn(a.z * rr * w.z));
                v[4 * c + 3] = __half2float(__float2half_rn(a.w * rr * w.w));
            }
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint4 u = *reinterpret_cast<const uint4*>(p.x16 + base + 8 * c);
                const float2 f0 = __half22float2(h2(u.x)), f1 = __half22float2(h2(u.y));
                const float2 f2 = __half22float2(h2(u.z)), f3 = __half22float2(h2(u.w));
                v[8 * c + 0] = f0.x; v[8 * c + 1] = f0.y; v[8 * c + 2] = f1.x; v[8 * c + 3] = f1.y;
                v[8 * c + 4] = f2.x; v[8 * c + 5] = f2.y; v[8 * c + 6] = f3.x; v[8 * c + 7] = f3.y;
            }
        }
        float lo = 0.f, hi = 0.f;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const __half2 p0 = __floats2half2_rn(v[4 * t], v[4 * t + 2]);
            const __half2 p1 = __floats2half2_rn(v[4 * t + 1], v[4 * t + 3]);
            const __half2 p2 = __floats2half2_rn(v[16 + 4 * t] * 0.0625f, v[18 + 4 * t] * 0.0625f);
            const __half2 p3 = __floats2half2_rn(v[17 + 4 * t] * 0.0625f, v[19 + 4 * t] * 0.0625f);
            const float2 f0 = __half22float2(p0), f1 = __half22float2(p1);
            const float2 f2 = __half22float2(p2), f3 = __half22float2(p3);
            lo += (f0.x + f0.y) + (f1.x + f1.y);
            hi += (f2.x + f2.y) + (f3.x + f3.y);
            xs[b * p.cstride + 4 * j + t] = make_uint4(u32(p0), u32(p1), u32(p2), u32(p3));
        }
        // sum (1024 + q) x_lo + (1024 + 16 q) x_hi/16 = sum (q - 8) x + 1032 sum x_lo + 1152 sum x_hi/16
        bias[j * 8 + b] = -(1032.0f * lo + 1152.0f * hi);
    }
}

__device__ __forceinline__ void store_out(const KParams& p, int n, int row, float v) {
    const size_t o = (size_t)n * p.y_ld + row;
    if (p.epilogue == QL_EPI_ADD_RESIDUAL) v += p.residual[o];
    if (p.y_dtype == QL_DTYPE_F16)
        reinterpret_cast<__half*>(p.y)[o] = __float2half_rn(v);
    else
        reinterpret_cast<float*>(p.y)[o] = v;
}

// Combine the K segments of a tile, apply the epilogue and (argmax) reduce the keys.
// Every thread of the CTA calls this (it contains CTA barriers).
__device__ __forceinline__ void finish_tile(const KParams& p, float* red, unsigned long long (*kred)[8],
                                            int tile, int seg, float (&acc)[4], bool oka, bool okb) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const bool silu_mul = (p.epilogue == QL_EPI_SILU_MUL);
    if (!oka) acc[0] = acc[1] = 0.f;
    if (!okb) acc[2] = acc[3] = 0.f;

    // combine the K segments of a tile
    if (p.S > 1) {
        float4* r4 = reinterpret_cast<float4*>(red);
        r4[warp * 32 + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        __syncthreads();
        if (seg == 0) {
            for (int s2 = 1; s2 < p.S; ++s2) {
                const float4 o = r4[(warp + s2) * 32 + lane];
                acc[0] += o.x; acc[1] += o.y; acc[2] += o.z; acc[3] += o.w;
            }
        }
    }

    unsigned long long best0 = 0ull, best1 = 0ull;   // argmax keys of columns 2t, 2t+1
    const int n0 = 2 * t, n1 = 2 * t + 1;
    if (seg == 0 && tile < p.ntile) {
        if (silu_mul) {
            const int i = tile * 8 + g;
            if (oka) {
                if (n0 < p.batch) store_out(p, n0, i, silu(acc[0]) * acc[2]);
                if (n1 < p.batch) store_out(p, n1, i, silu(acc[1]) * acc[3]);
            }
        } else if (p.epilogue == kEpiArgmax) {
            const int rga = tile * 16 + g, rgb = rga + 8;
            if (oka) {
                if (n0 < p.batch) {
                    best0 = argmax_key(acc[0], rga);
                    if (p.y) reinterpret_cast<float*>(p.y)[(size_t)n0 * p.y_ld + rga] = acc[0];
                }
                if (n1 < p.batch) {
                    best1 = argmax_key(acc[1], rga);
                    if (p.y) reinterpret_cast<float*>(p.y)[(size_t)n1 * p.y_ld + rga] = acc[1];
                }
            }
            if (okb) {
                if (n0 < p.batch) {
                    const unsigned long long k = argmax_key(acc[2], rgb);
                    best0 = k > best0 ? k : best0;
                    if (p.y) reinterpret_cast<float*>(p.y)[(size_t)n0 * p.y_ld + rgb] = acc[2];
                }
                if (n1 < p.batch) {
                    const unsigned long long k = argmax_key(acc[3], rgb);
                    best1 = k > best1 ? k : best1;
                    if (p.y) reinterpret_cast<float*>(p.y)[(size_t)n1 * p.y_ld + rgb] = acc[3];
                }
            }
        } else {
            const int rga = tile * 16 + g, rgb = rga + 8;
            if (oka) {
                if (n0 < p.batch) store_out(p, n0, rga, acc[0]);
                if (n1 < p.batch) store_out(p, n1, rga, acc[1]);
            }
            if (okb) {
                if (n0 < p.batch) store_out(p, n0, rgb, acc[2]);
                if (n1 < p.batch) store_out(p, n1, rgb, acc[3]);
            }
        }
    }
    if (p.epilogue == kEpiArgmax) {
        // lanes with the same t hold the same two columns: reduce over g, then over warps
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            const unsigned long long k0 = __shfl_xor_sync(0xffffffffu, best0, o);
            const unsigned long long k1 = __shfl_xor_sync(0xffffffffu, best1, o);
            best0 = k0 > best0 ? k0 : best0;
            best1 = k1 > best1 ? k1 : best1;
        }
        if (lane < 4) {
            kred[warp][2 * lane] = best0;
            kred[warp][2 * lane + 1] = best1;
        }
        __syncthreads();
        if (threadIdx.x < 8 && (int)threadIdx.x < p.batch) {
            const int b = threadIdx.x;
            unsigned long long m = 0ull;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) m = kred[w][b] > m ? kred[w][b] : m;
            const bool act = p.active == nullptr || p.active[b] != 0;
            if (m && act) atomicMax(p.keys + b, m);
        }
    }
}

__global__ void __launch_bounds__(kThreads, 3) gemv_q4_0_mma_kernel(KParams p, DevError* err) {
    extern __shared__ __align__(16) unsigned char smem[];
    uint4* xs = reinterpret_cast<uint4*>(smem);
    float* bias = reinterpret_cast<float*>(xs + (size_t)p.batch * p.cstride);
    float* red = bias + (size_t)p.nblk * 8;           // [kWarps][32][4]
    __shared__ unsigned long long kred[kWarps][8];
    (void)err;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const bool silu_mul = (p.epilogue == QL_EPI_SILU_MUL);
    const int half_rows = p.rows >> 1;
    const int tiles_per_cta = kWarps / p.S;
    const int tile = blockIdx.x * tiles_per_cta + warp / p.S;
    const int seg = warp % p.S;

    // The weights do not depend on the previous kernel: warm L2 with this CTA's first codes
    // while the predecessor drains.
    if (threadIdx.x == 0) {
        const size_t row_bytes = (size_t)p.nblk * 16;
        const int t0 = blockIdx.x * tiles_per_cta;
        const int nt = min(tiles_per_cta, p.ntile - t0);
        if (nt > 0) {
            const int rows_per_tile = silu_mul ? 8 : 16;
            const int limit = silu_mul ? half_rows : p.rows;
            const int r0 = t0 * rows_per_tile;
            size_t bytes = row_bytes * (size_t)min(nt * rows_per_tile, limit - r0);
            bytes = bytes > 49152 ? 49152 : bytes;
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.quants + (size_t)r0 * row_bytes),
                         "r"((uint32_t)bytes) : "memory");
            if (silu_mul)
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                             ::"l"(p.quants + (size_t)(half_rows + r0) * row_bytes), "r"((uint32_t)bytes)
                             : "memory");
        }
    }
    pdl_wait();
    stage_x(p, xs, bias, red);
    __syncthreads();
    pdl_trigger();

    // rows of this lane: ra (fragment row g) and rb (row g + 8)
    int ra, rb;
    bool oka, okb;
    if (silu_mul) {
        const int i = tile * 8 + g;
        oka = okb = (tile < p.ntile) && i < half_rows;
        ra = oka ? i : 0;
        rb = okb ? half_rows + i : 0;
    } else {
        ra = tile * 16 + g;
        rb = ra + 8;
        oka = (tile < p.ntile) && ra < p.rows;
        okb = (tile < p.ntile) && rb < p.rows;
        ra = oka ? ra : 0;
        rb = okb ? rb : 0;
    }
    const int j0 = seg * p.seg_blocks;
    const int j1 = (tile < p.ntile) ? min(p.nblk, j0 + p.seg_blocks) : j0;
    const int nit = j1 > j0 ? j1 - j0 : 0;
    const uint32_t* qa = reinterpret_cast<const uint32_t*>(p.quants) + ((size_t)ra * p.nblk + j0) * 4 + t;
    const uint32_t* qb = reinterpret_cast<const uint32_t*>(p.quants) + ((size_t)rb * p.nblk + j0) * 4 + t;
    const unsigned short* sa = reinterpret_cast<const unsigned short*>(p.scales) + (size_t)ra * p.nblk + j0;
    const unsigned short* sb = reinterpret_cast<const unsigned short*>(p.scales) + (size_t)rb * p.nblk + j0;
    const bool has_col = g < p.batch;
    const uint4* xcol = xs + (size_t)(has_col ? g : 0) * p.cstride;

    uint32_t rwa[kD], rwb[kD], rsc[kD];
#pragma unroll
    for (int u = 0; u < kD; ++u) {
        if (u < nit) {
            rwa[u] = __ldg(qa + 4 * u);
            rwb[u] = __ldg(qb + 4 * u);
            rsc[u] = (uint32_t)__ldg(sa + u) | ((uint32_t)__ldg(sb + u) << 16);
        }
    }
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int it0 = 0; it0 < nit; it0 += kD) {
#pragma unroll
        for (int u = 0; u < kD; ++u) {
            const int it = it0 + u;
            if (it < nit) {
                const int j = j0 + it;
                const uint32_t wa = rwa[u], wb = rwb[u];
                const __half2 sc = h2(rsc[u]);
                const int nx = it + kD;
                if (nx < nit) {
                    rwa[u] = __ldg(qa + 4 * nx);
                    rwb[u] = __ldg(qb + 4 * nx);
                    rsc[u] = (uint32_t)__ldg(sa + nx) | ((uint32_t)__ldg(sb + nx) << 16);
                }
                uint4 X = has_col ? xcol[4 * j + t] : make_uint4(0u, 0u, 0u, 0u);
                const float2 bz = *reinterpret_cast<const float2*>(bias + j * 8 + 2 * t);
                float c[4] = {bz.x, bz.y, bz.x, bz.y};
                const uint32_t sa8 = wa >> 8, sb8 = wb >> 8;
                mma16816(c, (wa & 0x000F000Fu) | 0x64006400u, (wb & 0x000F000Fu) | 0x64006400u,
                         (sa8 & 0x000F000Fu) | 0x64006400u, (sb8 & 0x000F000Fu) | 0x64006400u, X.x, X.y);
                mma16816(c, (wa & 0x00F000F0u) | 0x64006400u, (wb & 0x00F000F0u) | 0x64006400u,
                         (sa8 & 0x00F000F0u) | 0x64006400u, (sb8 & 0x00F000F0u) | 0x64006400u, X.z, X.w);
                const float2 d = __half22float2(sc);
                acc[0] = fmaf(d.x, c[0], acc[0]);
                acc[1] = fmaf(d.x, c[1], acc[1]);
                acc[2] = fmaf(d.y, c[2], acc[2]);
                acc[3] = fmaf(d.y, c[3], acc[3]);
            }
        }
    }
    finish_tile(p, red, kred, tile, seg, acc, oka, okb);
}


// ---------------------------------------------------------------------------------------------
// The same GEMV with the codes streamed into shared memory by the bulk-copy engine. Each warp
// owns a ring of NS stages; a stage holds 8 blocks (256 k) of its 16 rows: 128 code bytes per
// row (rows padded to 144 B so the 8 row-lanes of a load hit distinct banks) and 16 scale bytes
// per row. Lanes 0..15 each issue the two copies of one row; completion is tracked by one
// mbarrier per stage (expect-tx bytes). The first NS stages are issued before the kernel waits
// on its predecessor, so the weight stream starts while the previous kernel drains.
constexpr int kStageBlocks = 8;
constexpr int kRowPitch = 144;
constexpr int kStageBytes = 16 * kRowPitch + 16 * 16;   // codes + scales of 16 rows
constexpr long long kSpinLimit = 1ll << 26;             // bounded mbarrier waits

__device__ __forceinline__ uint32_t smem_u32(const void* ptr) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    for (long long i = 0; i < kSpinLimit; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
    }
    return false;
}

// Issue the copies of one stage: lane r < 16 copies row r's 128 code bytes and 16 scale bytes.
__device__ __forceinline__ void issue_stage(const KParams& p, uint32_t ring, uint32_t bar, int lane,
                                            int row_r, bool ok_r, int jblk, uint32_t bytes) {
    if (lane == 0)
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
    __syncwarp();
    if (lane < 16 && ok_r) {
        const uint8_t* src = p.quants + ((size_t)row_r * p.nblk + jblk) * 16;
        const __half* ssrc = p.scales + (size_t)row_r * p.nblk + jblk;
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], 128, [%2];"
            ::"r"(ring + lane * kRowPitch), "l"(src), "r"(bar) : "memory");
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], 16, [%2];"
            ::"r"(ring + 16 * kRowPitch + lane * 16), "l"(ssrc), "r"(bar) : "memory");
    }
}

__global__ void __launch_bounds__(kThreads, 2) gemv_q4_0_bulk_kernel(KParams p, int NS, DevError* err) {
    extern __shared__ __align__(16) unsigned char smem[];
    // layout: rings | mbarriers | xs | bias | red
    unsigned char* rings = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(rings + (size_t)kWarps * NS * kStageBytes);
    uint4* xs = reinterpret_cast<uint4*>(bars + kWarps * NS);
    float* bias = reinterpret_cast<float*>(xs + (size_t)p.batch * p.cstride);
    float* red = bias + (size_t)p.nblk * 8;
    __shared__ unsigned long long kred[kWarps][8];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const bool silu_mul = (p.epilogue == QL_EPI_SILU_MUL);
    const int half_rows = p.rows >> 1;
    const int tiles_per_cta = kWarps / p.S;
    const int tile = blockIdx.x * tiles_per_cta + warp / p.S;
    const int seg = warp % p.S;
    const bool live = tile < p.ntile;

    // the weight row each lane copies (lanes 0..15 -> tile rows 0..15)
    const int rr = lane & 15;
    int row_r;
    bool ok_r;
    if (silu_mul) {
        const int i = tile * 8 + (rr & 7);
        ok_r = live && i < half_rows;
        row_r = rr < 8 ? i : half_rows + i;
    } else {
        row_r = tile * 16 + rr;
        ok_r = live && row_r < p.rows;
    }
    // bytes one stage delivers: 144 per valid row
    uint32_t valid = __ballot_sync(0xffffffffu, lane < 16 && ok_r);
    const uint32_t stage_bytes = (uint32_t)__popc(valid) * (128u + 16u);

    const uint32_t ring0 = smem_u32(rings + (size_t)warp * NS * kStageBytes);
    const uint32_t bar0 = smem_u32(bars + warp * NS);
    if (lane == 0) {
        for (int s2 = 0; s2 < NS; ++s2)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar0 + 8 * s2) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    const int j0 = seg * p.seg_blocks;
    const int nst = live ? p.seg_blocks / kStageBlocks : 0;
    // weights do not depend on the previous kernel: start streaming before the PDL wait
    for (int s2 = 0; s2 < NS && s2 < nst; ++s2)
        issue_stage(p, ring0 + s2 * kStageBytes, bar0 + 8 * s2, lane, row_r, ok_r, j0 + s2 * kStageBlocks,
                    stage_bytes);

    pdl_wait();
    stage_x(p, xs, bias, red);
    __syncthreads();
    pdl_trigger();

    const bool has_col = g < p.batch;
    const uint4* xcol = xs + (size_t)(has_col ? g : 0) * p.cstride;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    bool failed = false;
    for (int st = 0; st < nst; ++st) {
        const int slot = st % NS;
        const uint32_t ring = ring0 + slot * kStageBytes, bar = bar0 + 8 * slot;
        // every lane observes the phase (visibility of the copied bytes); the decision is uniform
        const bool ok = __all_sync(0xffffffffu, mbar_wait(bar, (uint32_t)((st / NS) & 1)));
        if (!ok) {
            failed = true;
            break;
        }
        const unsigned char* rs = rings + (size_t)(warp * NS + slot) * kStageBytes;
        const uint32_t* ca = reinterpret_cast<const uint32_t*>(rs + g * kRowPitch) + t;
        const uint32_t* cb = reinterpret_cast<const uint32_t*>(rs + (g + 8) * kRowPitch) + t;
        const unsigned short* sca = reinterpret_cast<const unsigned short*>(rs + 16 * kRowPitch + g * 16);
        const unsigned short* scb = reinterpret_cast<const unsigned short*>(rs + 16 * kRowPitch + (g + 8) * 16);
        const int jb = j0 + st * kStageBlocks;
#pragma unroll
        for (int jj = 0; jj < kStageBlocks; ++jj) {
            const uint32_t wa = ca[4 * jj], wb = cb[4 * jj];
            const float da = __half2float(__ushort_as_half(sca[jj]));
            const float db = __half2float(__ushort_as_half(scb[jj]));
            const int j = jb + jj;
            const uint4 X = has_col ? xcol[4 * j + t] : make_uint4(0u, 0u, 0u, 0u);
            const float2 bz = *reinterpret_cast<const float2*>(bias + j * 8 + 2 * t);
            float c[4] = {bz.x, bz.y, bz.x, bz.y};
            const uint32_t sa8 = wa >> 8, sb8 = wb >> 8;
            mma16816(c, (wa & 0x000F000Fu) | 0x64006400u, (wb & 0x000F000Fu) | 0x64006400u,
                     (sa8 & 0x000F000Fu) | 0x64006400u, (sb8 & 0x000F000Fu) | 0x64006400u, X.x, X.y);
            mma16816(c, (wa & 0x00F000F0u) | 0x64006400u, (wb & 0x00F000F0u) | 0x64006400u,
                     (sa8 & 0x00F000F0u) | 0x64006400u, (sb8 & 0x00F000F0u) | 0x64006400u, X.z, X.w);
            acc[0] = fmaf(da, c[0], acc[0]);
            acc[1] = fmaf(da, c[1], acc[1]);
            acc[2] = fmaf(db, c[2], acc[2]);
            acc[3] = fmaf(db, c[3], acc[3]);
        }
        __syncwarp();
        if (st + NS < nst) {
            // the slot's generic-proxy reads are done; order them before the async-proxy refill
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue_stage(p, ring, bar, lane, row_r, ok_r, j0 + (st + NS) * kStageBlocks, stage_bytes);
        }
    }
    if (failed && lane == 0) record_device_error(err, kErrGemvStage, tile, seg);
    // fragment rows of this lane
    bool oka, okb;
    if (silu_mul) {
        oka = okb = live && tile * 8 + g < half_rows;
    } else {
        oka = live && tile * 16 + g < p.rows;
        okb = live && tile * 16 + g + 8 < p.rows;
    }
    finish_tile(p, red, kred, tile, seg, acc, oka, okb);
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
    cudaError_t e = cudaFuncSetAttribute(gemv_q4_0_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kMaxStageBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemv_q4_0_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
    if (e != cudaSuccess) return cuda_error(e, "gemv: cudaFuncSetAttribute");
    done.insert(dev);
    return QL_OK;
}

int gemv_launch(const GemvArgs& a, cudaStream_t s, bool pdl) {
    QL_REQUIRE(a.scales && a.quants && a.y, "gemv: null pointer");
    QL_REQUIRE(a.rows > 0 && a.cols > 0 && a.cols % 32 == 0, "gemv: need rows > 0, cols % 32 == 0");
    QL_REQUIRE(a.rows < (1ll << 31) && a.cols < (1ll << 24) && a.rows * (a.cols / 32) < (1ll << 29),
               "gemv: matrix too large");
    QL_REQUIRE(a.batch >= 1 && a.batch <= 64, "gemv: batch must be in [1, 64]");
    QL_REQUIRE(a.prologue == kProX16 ? a.x16 != nullptr : (a.xf && a.norm_w), "gemv: null input");
    QL_REQUIRE(a.epilogue != QL_EPI_SILU_MUL || a.rows % 2 == 0, "gemv: silu_mul needs even rows");
    QL_REQUIRE(a.epilogue != QL_EPI_ADD_RESIDUAL || (a.residual && a.y_dtype == QL_DTYPE_F32),
               "gemv: residual epilogue needs an f32 residual and f32 output");
    QL_REQUIRE(a.epilogue != kEpiArgmax || a.argmax_keys, "gemv: argmax needs key buffer");
    QL_REQUIRE(a.y_dtype == QL_DTYPE_F32 || a.y_dtype == QL_DTYPE_F16, "gemv: bad y dtype");
    QL_REQUIRE(a.epilogue != kEpiArgmax || a.y_dtype == QL_DTYPE_F32, "gemv: argmax logits are f32");
    auto al = [](const void* q, uintptr_t n) { return (reinterpret_cast<uintptr_t>(q) & (n - 1)) == 0; };
    QL_REQUIRE(al(a.quants, 16) && al(a.scales, 4) && al(a.x16, 16) && al(a.xf, 16) && al(a.norm_w, 16) &&
                   al(a.y, 4) && al(a.residual, 4),
               "gemv: codes, activations and norm weights must be 16-byte aligned, scales and outputs 4-byte");
    if (!device_error_record()) return set_error(QL_ECUDA, "gemv: no device error record");
    if (int rc = gemv_prepare()) return rc;

    const int nblk = (int)(a.cols / 32);
    const int cstride = nblk * 4 + 4;                              // +64 B: no bank aliasing
    const size_t fixed = (size_t)nblk * 8 * 4 + kWarps * 32 * 16;  // bias + segment reduction
    QL_REQUIRE(fixed + (size_t)cstride * 16 <= kMaxStageBytes, "gemv: cols too large for the staged activation");
    int nb_max = (int)((kMaxStageBytes - fixed) / ((size_t)cstride * 16));
    if (nb_max > 8) nb_max = 8;
    const bool silu = a.epilogue == QL_EPI_SILU_MUL;
    const int out_ld = (int)(silu ? a.rows / 2 : a.rows);
    const int sms = num_sms();

    for (int b0 = 0; b0 < a.batch; b0 += nb_max) {
        const int nb = a.batch - b0 < nb_max ? a.batch - b0 : nb_max;
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
        p.ntile = silu ? (int)((a.rows / 2 + 7) / 8) : (int)((a.rows + 15) / 16);
        p.cstride = cstride;
        const size_t stage_smem = fixed + (size_t)nb * cstride * 16;
        // The bulk-copy kernel needs whole 8-block stages and 16-byte aligned scale rows.
        const bool bulk = nblk % kStageBlocks == 0 && (reinterpret_cast<uintptr_t>(a.scales) & 15) == 0;
        int S = 1;
        cudaError_t e;
        if (bulk) {
            // split K over the warps of a CTA until the grid holds ~3 warps per SM sub-partition,
            // keeping whole stages and at least two of them per segment
            while (S < kWarps && (long long)p.ntile * S < 12ll * sms && nblk % (16 * S) == 0 &&
                   nblk / (2 * S) >= 2 * kStageBlocks)
                S *= 2;
            p.S = S;
            p.seg_blocks = nblk / S;
            const size_t per_stage = (size_t)kWarps * (kStageBytes + 8);
            int NS = (int)(((size_t)113 * 1024 - stage_smem) / per_stage);
            NS = NS > 4 ? 4 : NS < 2 ? 2 : NS;
            const size_t smem = (size_t)NS * per_stage + stage_smem;
            const int grid = (p.ntile + kWarps / S - 1) / (kWarps / S);
            e = launch(gemv_q4_0_bulk_kernel, dim3(grid), dim3(kThreads), smem, s, pdl, p, NS,
                       device_error_record());
        } else {
            while (S < kWarps && (long long)p.ntile * S < 12ll * sms && nblk / (2 * S) >= 8) S *= 2;
            p.S = S;
            p.seg_blocks = (nblk + S - 1) / S;
            const int grid = (p.ntile + kWarps / S - 1) / (kWarps / S);
            e = launch(gemv_q4_0_mma_kernel, dim3(grid), dim3(kThreads), stage_smem, s, pdl, p,
                       device_error_record());
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
