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

#include <cstdlib>
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

// SiLU with the fast exponential and division (the result is rounded to f16)
__device__ __forceinline__ float silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

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
    NextWeights next;  // weights of the following kernel, prefetched into L2
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
            const float r = rsqrtf(fmaf(t, 1.0f / (float)cols, p.eps));
#pragma unroll
            for (int bb = 0; bb < 8; ++bb)
                if (bb == b) rs[bb] = r;
        }
        __syncthreads();   // red is reused later
    }
    // one item = one 16-byte chunk (column b, block j, lane slot t); the 4 chunks of a block are
    // handled by 4 consecutive threads, which reduce the block's offset term with shuffles
    // columns past the batch contribute nothing: their offset terms are zero
    for (int i = tid; i < (8 - p.batch) * p.nblk; i += kThreads) {
        const int b = p.batch + i / p.nblk, j = i % p.nblk;
        bias[j * 8 + b] = 0.f;
    }
    // the loop bound is warp-uniform (whole warps iterate together) because of the shuffles
    const int nitems = p.batch * p.nblk * 4;
    for (int wbase = tid & ~31; wbase < nitems; wbase += kThreads) {
        const int item = wbase + (tid & 31);
        const int t = item & 3, bj = item >> 2;
        const int b = bj / p.nblk, j = bj - b * p.nblk;
        float lo[4] = {0.f, 0.f, 0.f, 0.f}, hi[4] = {0.f, 0.f, 0.f, 0.f};
        if (item < nitems) {
            const size_t off = (size_t)b * cols + 32 * j + 4 * t;
            if (p.prologue == kProRmsF32) {
                float rr = rs[0];
#pragma unroll
                for (int bb = 1; bb < 8; ++bb)
                    if (bb == b) rr = rs[bb];
                const float4 a4 = *reinterpret_cast<const float4*>(p.xf + off);
                const float4 h4 = *reinterpret_cast<const float4*>(p.xf + off + 16);
                const float4 wa = *reinterpret_cast<const float4*>(p.norm_w + 32 * j + 4 * t);
                const float4 wh = *reinterpret_cast<const float4*>(p.norm_w + 32 * j + 16 + 4 * t);
                lo[0] = a4.x * rr * wa.x; lo[1] = a4.y * rr * wa.y; lo[2] = a4.z * rr * wa.z; lo[3] = a4.w * rr * wa.w;
                hi[0] = h4.x * rr * wh.x; hi[1] = h4.y * rr * wh.y; hi[2] = h4.z * rr * wh.z; hi[3] = h4.w * rr * wh.w;
            } else {
                const uint2 a2 = *reinterpret_cast<const uint2*>(p.x16 + off);
                const uint2 h2v = *reinterpret_cast<const uint2*>(p.x16 + off + 16);
                const float2 f0 = __half22float2(h2(a2.x)), f1 = __half22float2(h2(a2.y));
                const float2 f2 = __half22float2(h2(h2v.x)), f3 = __half22float2(h2(h2v.y));
                lo[0] = f0.x; lo[1] = f0.y; lo[2] = f1.x; lo[3] = f1.y;
                hi[0] = f2.x; hi[1] = f2.y; hi[2] = f3.x; hi[3] = f3.y;
            }
        }
        // activations rounded to f16 (the GEMV's input precision); high ones pre-divided by 16
        const __half2 p0 = __floats2half2_rn(lo[0], lo[2]);
        const __half2 p1 = __floats2half2_rn(lo[1], lo[3]);
        const __half2 p2 = __floats2half2_rn(__half2float(__float2half_rn(hi[0])) * 0.0625f,
                                             __half2float(__float2half_rn(hi[2])) * 0.0625f);
        const __half2 p3 = __floats2half2_rn(__half2float(__float2half_rn(hi[1])) * 0.0625f,
                                             __half2float(__float2half_rn(hi[3])) * 0.0625f);
        const float2 f0 = __half22float2(p0), f1 = __half22float2(p1);
        const float2 f2 = __half22float2(p2), f3 = __half22float2(p3);
        // sum (1024 + q) x_lo + (1024 + 16 q) x_hi/16 = sum (q - 8) x + 1032 sum x_lo + 1152 sum x_hi/16
        float part = 1032.0f * ((f0.x + f0.y) + (f1.x + f1.y)) + 1152.0f * ((f2.x + f2.y) + (f3.x + f3.y));
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        if (item < nitems) {
            xs[b * p.cstride + 4 * j + t] = make_uint4(u32(p0), u32(p1), u32(p2), u32(p3));
            if (t == 0) bias[j * 8 + b] = -part;
        }
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
    l2_prefetch_share(p.next.ptr[0], p.next.bytes[0]);
    l2_prefetch_share(p.next.ptr[1], p.next.bytes[1]);
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
// The main GEMV kernel (K % 128 == 0). Each warp streams its tile through a ring of kStages
// shared-memory stages filled by 16-byte asynchronous copies (cp.async, L2 only): a stage holds 4
// blocks x 16 rows of codes (1 KB; lane l copies block l >> 3 of tile rows (l & 7) and (l & 7) + 8)
// and the 16 rows' 4 f16 scales (128 B). No registers are held by loads in flight, so a warp keeps
// kStages KB outstanding; the first stages are issued before the kernel waits on its predecessor.
// An 8x8 b16 ldmatrix tile is 8 rows of 16 bytes - one q4_0 block per row - so two ldmatrix.x4 per
// stage hand every lane exactly the 32-bit code words its MMA fragments need (word t of block j
// for rows g and g + 8).
constexpr int kGroupBlocks = 4;
constexpr int kStages = 6;
constexpr int kStageBytes = kGroupBlocks * 16 * 16 + 16 * 8;   // codes + scales of one stage

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__global__ void __launch_bounds__(kThreads, 3) gemv_q4_0_lsm_kernel(KParams p, DevError* err) {
    extern __shared__ __align__(16) unsigned char smem[];
    // layout: per-warp rings (kStages x kStageBytes) | xs | bias | red
    unsigned char* rings = smem;
    uint4* xs = reinterpret_cast<uint4*>(rings + (size_t)kWarps * kStages * kStageBytes);
    float* bias = reinterpret_cast<float*>(xs + (size_t)p.batch * p.cstride);
    float* red = bias + (size_t)p.nblk * 8;
    __shared__ unsigned long long kred[kWarps][8];
    (void)err;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const bool silu_mul = (p.epilogue == QL_EPI_SILU_MUL);
    const int half_rows = p.rows >> 1;
    const int tiles_per_cta = kWarps / p.S;
    const int seg = warp % p.S;
    // The CTA walks tile groups blockIdx.x, blockIdx.x + gridDim.x, ...; every warp runs the same
    // number of (tile, segment) tasks, so the per-task barriers line up.
    const int ngroups = (p.ntile + tiles_per_cta - 1) / tiles_per_cta;
    const int my_groups = (int)blockIdx.x < ngroups ? (ngroups - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
    const int nit = p.seg_blocks / kGroupBlocks;      // iterations (4 blocks each) per task
    const int total = my_groups * nit;
    const int j0 = seg * p.seg_blocks;
    const int lr = lane & 7, lb = lane >> 3;

    auto tile_of = [&](int grp) { return ((int)blockIdx.x + grp * (int)gridDim.x) * tiles_per_cta + warp / p.S; };
    // global row of tile row r (invalid rows read row 0; their results are discarded)
    auto tile_row = [&](int tile, int r, bool& ok) -> int {
        const bool live = tile < p.ntile;
        if (silu_mul) {
            const int i = tile * 8 + (r & 7);
            ok = live && i < half_rows;
            return ok ? (r < 8 ? i : half_rows + i) : 0;
        }
        const int row = tile * 16 + r;
        ok = live && row < p.rows;
        return ok ? row : 0;
    };
    const uint32_t ring_s = static_cast<uint32_t>(__cvta_generic_to_shared(rings)) +
                            (uint32_t)(warp * kStages * kStageBytes);
    const uint32_t dA = (uint32_t)((lb * 16 + lr) * 16), dB = dA + 8 * 16;
    const uint32_t dS = (uint32_t)(kGroupBlocks * 16 * 16 + (lane & 15) * 8);

    // load cursor: (group, iteration) of the next stage to issue, and its source pointers
    int l_grp = 0, l_it = 0;
    const uint8_t* srcA = nullptr;
    const uint8_t* srcB = nullptr;
    const __half* srcS = nullptr;
    auto set_task = [&](int grp) {
        bool ok;
        const int tile = tile_of(grp);
        const int rowA = tile_row(tile, lr, ok), rowB = tile_row(tile, lr + 8, ok);
        const int rowS = tile_row(tile, lane & 15, ok);
        srcA = p.quants + ((size_t)rowA * p.nblk + j0 + lb) * 16;
        srcB = p.quants + ((size_t)rowB * p.nblk + j0 + lb) * 16;
        srcS = p.scales + (size_t)rowS * p.nblk + j0;
    };
    set_task(0);
    auto issue = [&](int it) {
        if (it < total) {
            const uint32_t st = ring_s + (uint32_t)((it % kStages) * kStageBytes);
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(st + dA), "l"(srcA + l_it * kGroupBlocks * 16) : "memory");
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(st + dB), "l"(srcB + l_it * kGroupBlocks * 16) : "memory");
            if (lane < 16)
                asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(st + dS), "l"(srcS + l_it * kGroupBlocks) : "memory");
            if (++l_it == nit) {
                l_it = 0;
                if (++l_grp < my_groups) set_task(l_grp);
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    // the weights do not depend on the previous kernel: start streaming before the PDL wait
#pragma unroll 1
    for (int it = 0; it < kStages; ++it) issue(it);
    l2_prefetch_share(p.next.ptr[0], p.next.bytes[0]);
    l2_prefetch_share(p.next.ptr[1], p.next.bytes[1]);

    pdl_wait();
    stage_x(p, xs, bias, red);
    __syncthreads();
    pdl_trigger();

    // ldmatrix row address of this lane: matrix m = lane >> 3 -> (block m >> 1, rows (m & 1) * 8 + r)
    const int lm = lane >> 3, lrow = lane & 7;
    const uint32_t a_lo = (uint32_t)(((lm >> 1) * 16 + (lm & 1) * 8 + lrow) * 16);
    const uint32_t a_hi = a_lo + 2 * 16 * 16;      // blocks 2 and 3
    const bool has_col = g < p.batch;
    const uint4* xcol = xs + (size_t)(has_col ? g : 0) * p.cstride;

    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    int c_grp = 0, c_it = 0;
#pragma unroll 1
    for (int it = 0; it < total; ++it) {
        asm volatile("cp.async.wait_group %0;" ::"n"(kStages - 1) : "memory");
        __syncwarp();
        const uint32_t st = ring_s + (uint32_t)((it % kStages) * kStageBytes);
        uint32_t w[8];   // wa0, wb0, wa1, wb1, wa2, wb2, wa3, wb3
        ldsm_x4(st + a_lo, w[0], w[1], w[2], w[3]);
        ldsm_x4(st + a_hi, w[4], w[5], w[6], w[7]);
        const unsigned char* stg = rings + (size_t)(warp * kStages + it % kStages) * kStageBytes;
        const uint2 sca = *reinterpret_cast<const uint2*>(stg + kGroupBlocks * 16 * 16 + g * 8);
        const uint2 scb = *reinterpret_cast<const uint2*>(stg + kGroupBlocks * 16 * 16 + (g + 8) * 8);
        __syncwarp();
        issue(it + kStages);                         // refill this slot (the reads above are done)
        const float2 da01 = __half22float2(h2(sca.x)), da23 = __half22float2(h2(sca.y));
        const float2 db01 = __half22float2(h2(scb.x)), db23 = __half22float2(h2(scb.y));
        const float da[4] = {da01.x, da01.y, da23.x, da23.y};
        const float db[4] = {db01.x, db01.y, db23.x, db23.y};
#pragma unroll
        for (int q = 0; q < kGroupBlocks; ++q) {
            const int j = j0 + c_it * kGroupBlocks + q;
            const uint32_t wa = w[2 * q], wb = w[2 * q + 1];
            const uint4 X = has_col ? xcol[4 * j + t] : make_uint4(0u, 0u, 0u, 0u);
            const float2 bz = *reinterpret_cast<const float2*>(bias + j * 8 + 2 * t);
            float c[4] = {bz.x, bz.y, bz.x, bz.y};
            const uint32_t sa8 = wa >> 8, sb8 = wb >> 8;
            mma16816(c, (wa & 0x000F000Fu) | 0x64006400u, (wb & 0x000F000Fu) | 0x64006400u,
                     (sa8 & 0x000F000Fu) | 0x64006400u, (sb8 & 0x000F000Fu) | 0x64006400u, X.x, X.y);
            mma16816(c, (wa & 0x00F000F0u) | 0x64006400u, (wb & 0x00F000F0u) | 0x64006400u,
                     (sa8 & 0x00F000F0u) | 0x64006400u, (sb8 & 0x00F000F0u) | 0x64006400u, X.z, X.w);
            acc[0] = fmaf(da[q], c[0], acc[0]);
            acc[1] = fmaf(da[q], c[1], acc[1]);
            acc[2] = fmaf(db[q], c[2], acc[2]);
            acc[3] = fmaf(db[q], c[3], acc[3]);
        }
        if (++c_it == nit) {
            const int tile = tile_of(c_grp);
            bool oka, okb;
            (void)tile_row(tile, g, oka);
            (void)tile_row(tile, g + 8, okb);
            finish_tile(p, red, kred, tile, seg, acc, oka, okb);
            acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
            c_it = 0;
            ++c_grp;
        }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

}  // namespace

// CTAs per SM of the main GEMV grid (the CTAs loop over tile groups): 3, the occupancy limit of
// the kernel, measured fastest in the decode step (1 per SM, which would leave room for the next
// kernel to start early, was slower). QL_GEMV_CTAS_PER_SM overrides it for A/B measurements.
int gemv_ctas_per_sm() {
    static int v = [] {
        const char* e = std::getenv("QL_GEMV_CTAS_PER_SM");
        const int n = e ? std::atoi(e) : 3;
        return n < 1 ? 1 : n > 8 ? 8 : n;
    }();
    return v;
}

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
        e = cudaFuncSetAttribute(gemv_q4_0_lsm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kMaxStageBytes + kWarps * kStages * kStageBytes);
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
        if (b0 == 0) p.next = a.next;
        p.ntile = silu ? (int)((a.rows / 2 + 7) / 8) : (int)((a.rows + 15) / 16);
        p.cstride = cstride;
        const size_t stage_smem = fixed + (size_t)nb * cstride * 16;
        // The main kernel needs whole 4-block groups and 8-byte aligned scale rows.
        const bool main = nblk % kGroupBlocks == 0 && (reinterpret_cast<uintptr_t>(a.scales) & 7) == 0;
        int S = 1;
        cudaError_t e;
        if (main) {
            // split K over the warps of a CTA until the grid holds ~3 warps per SM sub-partition,
            // keeping whole groups and at least two groups per segment
            while (S < kWarps && (long long)p.ntile * S < 12ll * sms && nblk % (2 * kGroupBlocks * S) == 0 &&
                   nblk / (2 * S) >= 2 * kGroupBlocks)
                S *= 2;
            p.S = S;
            p.seg_blocks = nblk / S;
            const size_t smem = (size_t)kWarps * kStages * kStageBytes + stage_smem;
            int grid = (p.ntile + kWarps / S - 1) / (kWarps / S);
            const int cap = gemv_ctas_per_sm() * sms;
            if (grid > cap) grid = cap;
            e = launch(gemv_q4_0_lsm_kernel, dim3(grid), dim3(kThreads), smem, s, pdl, p, device_error_record());
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
