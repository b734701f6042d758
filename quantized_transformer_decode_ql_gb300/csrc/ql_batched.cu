// Batched q4_0 GEMV (batch 3-32) over the tile stream layout: every weight byte is streamed
// once per call, whatever the batch.
//
// [IL] inferencelayer cuda_llm.rs, CudaQwen3::gemv (the q4_0 format, one GEMV per projection
// group) at the batch sizes where it becomes a skinny GEMM: each weight is used batch times, so
// the products go to the tensor cores (mma.sync m16n8k16, f16 in, f32 accumulate) with the exact
// nibble expansion of the batch-1 kernel (1024 + q and 1024 + 16 q in the A fragment, offsets
// folded into the accumulator start, one FFMA per block and column for the f16 scale).
//
// Why this shape (GB300): the activations of all batch columns for the full K (32 columns x
// 12288 x f16 = 768 KB for the down projection) do not fit in shared memory next to the weight
// ring, and re-reading the weights per column group multiplies the step's dominant traffic. So
// K is cut into windows of 1024 (8 units per tile): the CTA stages one window of every column,
// its warps consume that window's units, then the CTA stages the next window. Within a group of
// up to 16 tiles, the units of a window are split over the 16 warps in the same way in every
// window, so each warp meets the same (at most two) tiles every time and keeps their
// accumulators in registers; tiles shared by warps are reduced in shared memory in warp order at
// the end of the group (deterministic). The weights arrive through the same per-warp ring of
// bulk copies (TMA) as the batch-1 kernel, in the order the windows consume them.
#include "ql_persist.cuh"

#include <cstdlib>
#include <mutex>
#include <set>

namespace ql {
namespace batched {

using persist::as_h2;
using persist::as_u32;
using persist::kSlotBytes;
using persist::kSlotUnits;
using persist::kStages;
using persist::kUnitBlocks;
using persist::kUnitBytes;

constexpr int kW = 16, kT = kW * 32;
constexpr int kWinUnits = 8;                       // units per tile per K window (1024 columns)
constexpr int kGroupTiles = 16;                    // tiles per group
constexpr int kMaxCols = 32;                       // batch columns per call
constexpr int kXStride = kWinUnits * kUnitBlocks * 4 + 4;   // uint4 per staged column (+64 B)
constexpr size_t kRing = (size_t)kW * kStages * kSlotBytes;
constexpr size_t kXBytes = (size_t)kMaxCols * kXStride * 16;   // one window of every column
constexpr size_t kPartBytes = (size_t)kW * 2 * 4 * 32 * 16;    // [warp][slot][n-tile][lane] float4
constexpr size_t kXPart = kXBytes > kPartBytes ? kXBytes : kPartBytes;
constexpr size_t kBiasBytes = (size_t)kWinUnits * kUnitBlocks * kMaxCols * 4;
constexpr size_t kSmem = kRing + kXPart + kBiasBytes;

struct BParams {
    PMat M;
    int B, epi, rms;
    const float* xf;       // rms: f32 [B][cols]
    const __half* x16;     // else f16 [B][cols]
    const float* norm_w;
    const float* rs_in;    // rms: [B] 1 / rms of each column (rms_stats_kernel)
    float eps;
    void* y;
    int ld;
    unsigned long long* keys;
    const int32_t* active;
    unsigned int* sync;    // [4]: [2] is the abort flag of the bounded waits
    DevError* err;
    unsigned long long timeout_ns;
};

// This CTA's tiles, K windows and groups.
struct Geo {
    int T0, T1, nst, kwu, nwin, ngroups;
};
__device__ __forceinline__ Geo geometry(const PMat& M) {
    Geo G;
    persist::cta_tiles(M.ntile, G.T0, G.T1);
    G.nst = M.nblk / kUnitBlocks;
    G.kwu = G.nst < kWinUnits ? G.nst : kWinUnits;
    G.nwin = G.nst / G.kwu;
    G.ngroups = (G.T1 - G.T0 + kGroupTiles - 1) / kGroupTiles;
    return G;
}
__device__ __forceinline__ int group_tiles(const Geo& G, int g) {
    const int t = G.T1 - G.T0 - kGroupTiles * g;
    return t < kGroupTiles ? t : kGroupTiles;
}
// This warp's units [a, b) of a (group, window): the same split in every window of a group.
__device__ __forceinline__ void warp_range(const Geo& G, int g, int warp, int& a, int& b) {
    const int U = group_tiles(G, g) * G.kwu;
    a = persist::warp_unit<kW>(U, warp);
    b = persist::warp_unit<kW>(U, warp + 1);
}

// Issue side of the ring: (group, window, unit) in consumption order; a copy never crosses a
// tile's run of kwu units.
struct BRing {
    int g, w, u, b;
    unsigned int issued, consumed;
    uint32_t base, mbar;
    int dead;
};
__device__ __forceinline__ void bring_seek(BRing& r, const Geo& G, int warp) {
    while (r.g < G.ngroups) {
        int a, b;
        warp_range(G, r.g, warp, a, b);
        if (a < b) {
            if (r.u < a || r.u >= b) r.u = a;
            r.b = b;
            return;
        }
        ++r.g;   // no units for this warp in the whole group
        r.w = 0;
        r.u = -1;
    }
}
__device__ __forceinline__ void bring_issue(BRing& r, const PMat& M, const Geo& G, int warp, int lane) {
    if (r.g >= G.ngroups || r.dead) return;
    const int tl = r.u / G.kwu, kk = r.u - tl * G.kwu;
    int n = r.b - r.u;
    n = n < kSlotUnits ? n : kSlotUnits;
    n = n < G.kwu - kk ? n : G.kwu - kk;
    if (lane == 0) {
        const int tile = G.T0 + kGroupTiles * r.g + tl, k = G.kwu * r.w + kk;
        const unsigned int slot = r.issued % kStages;
        const uint32_t mb = r.mbar + slot * 8, dst = r.base + slot * kSlotBytes;
        const uint32_t bytes = (uint32_t)(n * kUnitBytes);
        const uint8_t* src = M.stream + ((size_t)tile * G.nst + k) * kUnitBytes;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mb), "r"(bytes) : "memory");
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                     ::"r"(dst), "l"(src), "r"(bytes), "r"(mb) : "memory");
    }
    ++r.issued;
    r.u += n;
    if (r.u == r.b) {
        if (++r.w == G.nwin) {
            r.w = 0;
            ++r.g;
            r.u = -1;
        } else {
            int a, b;
            warp_range(G, r.g, warp, a, b);
            r.u = a;
        }
        bring_seek(r, G, warp);
    }
}

__device__ __forceinline__ void bring_wait(BRing& r, const BParams& p, unsigned int n) {
    if (r.dead) return;
    const uint32_t mb = r.mbar + (n % kStages) * 8, parity = (n / kStages) & 1u;
    for (int spin = 0; spin < persist::kFastSpins; ++spin)
        if (persist::mbar_test(mb, parity)) return;
    const unsigned long long t0 = persist::global_ns();
    for (unsigned int spin = 1;; ++spin) {
        if (persist::mbar_test(mb, parity)) return;
        if ((spin & 63u) == 0 && persist::global_ns() - t0 > p.timeout_ns) break;
    }
    if ((threadIdx.x & 31) == 0) {
        record_device_error(p.err, kErrGemvStage, blockIdx.x, (long long)n);
        atomicExch(p.sync + 2, 1u);
    }
    r.dead = 1;
}

// 1 / rms of every column (the RMSNorm statistics over the full K), computed once by
// rms_stats_kernel for all CTAs.
__device__ void load_column_rms(const BParams& p, float* rs) {
    if ((int)threadIdx.x < p.B) rs[threadIdx.x] = __ldcg(p.rs_in + threadIdx.x);
    __syncthreads();
}

// Stage window w of every column: f16 pairs in the order a code word expands to (high ones
// pre-divided by 16) and the accumulator start -(1032 sum x_lo + 1152 sum x_hi / 16) of every
// (block, column); columns past the batch have zero offsets (their activations are never read).
__device__ void stage_window(const BParams& p, const Geo& G, int w, const float* rs, uint4* xs, float* bias) {
    const int tid = threadIdx.x;
    const int nb = G.kwu * kUnitBlocks;        // blocks in the window
    const int cols = p.M.nblk * 32;
    const int j0 = w * nb;
    for (int i = tid; i < nb * kMaxCols; i += kT) bias[i] = 0.f;
    __syncthreads();
    const int nitems = p.B * nb * 4;
    constexpr int kChunk = 4;   // items per thread whose loads are in flight together
    for (int base = 0; base < nitems; base += kChunk * kT) {   // warp-uniform bounds (shuffles)
        float4 la[kChunk], lh[kChunk];
        uint2 ha[kChunk], hh[kChunk];
#pragma unroll
        for (int r = 0; r < kChunk; ++r) {
            const int item = base + r * kT + tid;
            if (item < nitems) {
                const int t = item & 3, cj = item >> 2, c = cj / nb, j = cj - c * nb;
                const size_t off = (size_t)c * cols + 32 * (j0 + j) + 4 * t;
                if (p.rms) {
                    la[r] = __ldcg(reinterpret_cast<const float4*>(p.xf + off));
                    lh[r] = __ldcg(reinterpret_cast<const float4*>(p.xf + off + 16));
                } else {
                    ha[r] = __ldcg(reinterpret_cast<const uint2*>(p.x16 + off));
                    hh[r] = __ldcg(reinterpret_cast<const uint2*>(p.x16 + off + 16));
                }
            }
        }
#pragma unroll
        for (int r = 0; r < kChunk; ++r) {
            if (base + r * kT >= nitems) break;   // warp-uniform
            const int item = base + r * kT + tid;
            const bool live = item < nitems;
            const int t = item & 3, cj = item >> 2, c = cj / nb, j = cj - c * nb;
            float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (live) {
                if (p.rms) {
                    const float4 wa = __ldg(reinterpret_cast<const float4*>(p.norm_w + 32 * (j0 + j) + 4 * t));
                    const float4 wh = __ldg(reinterpret_cast<const float4*>(p.norm_w + 32 * (j0 + j) + 16 + 4 * t));
                    const float rr = rs[c];
                    const float4 a = la[r], h = lh[r];
                    v[0] = a.x * rr * wa.x; v[1] = a.y * rr * wa.y; v[2] = a.z * rr * wa.z; v[3] = a.w * rr * wa.w;
                    v[4] = h.x * rr * wh.x; v[5] = h.y * rr * wh.y; v[6] = h.z * rr * wh.z; v[7] = h.w * rr * wh.w;
                } else {
                    const float2 f0 = __half22float2(as_h2(ha[r].x)), f1 = __half22float2(as_h2(ha[r].y));
                    const float2 f2 = __half22float2(as_h2(hh[r].x)), f3 = __half22float2(as_h2(hh[r].y));
                    v[0] = f0.x; v[1] = f0.y; v[2] = f1.x; v[3] = f1.y;
                    v[4] = f2.x; v[5] = f2.y; v[6] = f3.x; v[7] = f3.y;
                }
            }
            const __half2 p0 = __floats2half2_rn(v[0], v[2]);
            const __half2 p1 = __floats2half2_rn(v[1], v[3]);
            const __half2 p2 = __floats2half2_rn(__half2float(__float2half_rn(v[4])) * 0.0625f,
                                                 __half2float(__float2half_rn(v[6])) * 0.0625f);
            const __half2 p3 = __floats2half2_rn(__half2float(__float2half_rn(v[5])) * 0.0625f,
                                                 __half2float(__float2half_rn(v[7])) * 0.0625f);
            const float2 f0 = __half22float2(p0), f1 = __half22float2(p1);
            const float2 f2 = __half22float2(p2), f3 = __half22float2(p3);
            // sum (1024 + q) x_lo + (1024 + 16 q) x_hi/16 = sum (q - 8) x + 1032 sum x_lo + 1152 sum x_hi/16
            float part = 1032.0f * ((f0.x + f0.y) + (f1.x + f1.y)) + 1152.0f * ((f2.x + f2.y) + (f3.x + f3.y));
            part += __shfl_xor_sync(0xffffffffu, part, 1);
            part += __shfl_xor_sync(0xffffffffu, part, 2);
            if (live) {
                xs[(size_t)c * kXStride + 4 * j + t] = make_uint4(as_u32(p0), as_u32(p1), as_u32(p2), as_u32(p3));
                if (t == 0) bias[j * kMaxCols + c] = -part;
            }
        }
    }
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// Epilogue of one finished tile for this lane's fragment (rows g, g + 8; columns 8 nt + 2t, +1).
template <int NT>
__device__ __forceinline__ void finish_tile(const BParams& p, int tile, const float (&acc)[NT][4],
                                            unsigned long long* kred, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int c = nt * 8 + 2 * t + e;
            if (c >= p.B) continue;
            const float va = acc[nt][e], vb = acc[nt][2 + e];   // rows g and g + 8
            if (p.epi == QL_EPI_SILU_MUL) {
                const int i = tile * 8 + g;
                if (i < (p.M.rows >> 1))
                    static_cast<__half*>(p.y)[(size_t)c * p.ld + i] = __float2half_rn(persist::silu(va) * vb);
                continue;
            }
            float* yf = static_cast<float*>(p.y);
            const int ra = tile * 16 + g, rb = ra + 8;
            if (p.epi == QL_EPI_ADD_RESIDUAL) {
                if (ra < p.M.rows) yf[(size_t)c * p.ld + ra] = __ldcg(yf + (size_t)c * p.ld + ra) + va;
                if (rb < p.M.rows) yf[(size_t)c * p.ld + rb] = __ldcg(yf + (size_t)c * p.ld + rb) + vb;
            } else {
                unsigned long long best = 0ull;
                if (ra < p.M.rows) {
                    yf[(size_t)c * p.ld + ra] = va;
                    best = persist::argmax_key(va, ra);
                }
                if (rb < p.M.rows) {
                    yf[(size_t)c * p.ld + rb] = vb;
                    const unsigned long long k2 = persist::argmax_key(vb, rb);
                    best = k2 > best ? k2 : best;
                }
                if (p.epi == kEpiArgmax && best) atomicMax(kred + c, best);
            }
        }
    }
}

template <int NT>
__global__ void __launch_bounds__(kT, 1) gemv_batched_kernel(const __grid_constant__ BParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ __align__(8) unsigned long long mbar[kW * kStages];
    __shared__ unsigned long long kred[kMaxCols];
    __shared__ float rs[kMaxCols];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    uint4* xs = reinterpret_cast<uint4*>(smem + kRing);
    float4* part = reinterpret_cast<float4*>(smem + kRing);   // aliases xs between groups
    float* bias = reinterpret_cast<float*>(smem + kRing + kXPart);
    const PMat& M = p.M;
    const Geo G = geometry(M);

    if (lane == 0)
        for (int i = 0; i < kStages; ++i)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(
                             static_cast<uint32_t>(__cvta_generic_to_shared(&mbar[warp * kStages + i]))) : "memory");
    if (tid < kMaxCols) kred[tid] = 0ull;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();
    BRing r;
    r.g = 0;
    r.w = 0;
    r.u = -1;
    r.b = 0;
    r.issued = r.consumed = 0;
    r.dead = 0;
    r.base = static_cast<uint32_t>(__cvta_generic_to_shared(smem)) + (uint32_t)(warp * kStages * kSlotBytes);
    r.mbar = static_cast<uint32_t>(__cvta_generic_to_shared(&mbar[warp * kStages]));
    bring_seek(r, G, warp);
#pragma unroll 1
    for (int i = 0; i < kStages; ++i) bring_issue(r, M, G, warp, lane);
    pdl_wait();
    pdl_trigger();
    if (p.rms) load_column_rms(p, rs);

    const int lm = lane >> 3, lrow = lane & 7;
    const uint32_t a_lo = (uint32_t)(((lm >> 1) * 16 + (lm & 1) * 8 + lrow) * 16);
    const unsigned char* ring_g = smem + (size_t)warp * kStages * kSlotBytes;
#pragma unroll 1
    for (int gi = 0; gi < G.ngroups; ++gi) {
        int a, b;
        warp_range(G, gi, warp, a, b);
        const int tl0 = a < b ? a / G.kwu : 0, tl1 = a < b ? (b - 1) / G.kwu : 0;
        float acc0[NT][4], acc1[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc0[nt][i] = acc1[nt][i] = 0.f;
#pragma unroll 1
        for (int w = 0; w < G.nwin; ++w) {
            __syncthreads();   // the previous window's (or group's) readers of xs / part are done
            stage_window(p, G, w, rs, xs, bias);
            __syncthreads();
#pragma unroll 1
            for (int u = a; u < b;) {
                const int tl = u / G.kwu, kk = u - tl * G.kwu;
                int n = b - u;
                n = n < kSlotUnits ? n : kSlotUnits;
                n = n < G.kwu - kk ? n : G.kwu - kk;
                bring_wait(r, p, r.consumed);
                __syncwarp();
                const unsigned int slot = r.consumed % kStages;
#pragma unroll 1
                for (int i = 0; i < n; ++i) {
                    const uint32_t st = r.base + slot * kSlotBytes + i * kUnitBytes;
                    const unsigned char* stg = ring_g + (size_t)slot * kSlotBytes + (size_t)i * kUnitBytes;
                    uint32_t wv[8];
                    ldsm_x4(st + a_lo, wv[0], wv[1], wv[2], wv[3]);
                    ldsm_x4(st + a_lo + 2 * 16 * 16, wv[4], wv[5], wv[6], wv[7]);
                    const uint2 sca = *reinterpret_cast<const uint2*>(stg + 1024 + g * 8);
                    const uint2 scb = *reinterpret_cast<const uint2*>(stg + 1024 + (g + 8) * 8);
                    const float2 da01 = __half22float2(as_h2(sca.x)), da23 = __half22float2(as_h2(sca.y));
                    const float2 db01 = __half22float2(as_h2(scb.x)), db23 = __half22float2(as_h2(scb.y));
                    const float da[4] = {da01.x, da01.y, da23.x, da23.y};
                    const float db[4] = {db01.x, db01.y, db23.x, db23.y};
                    const bool first = tl == tl0;
#pragma unroll
                    for (int q = 0; q < kUnitBlocks; ++q) {
                        const int j = (kk + i) * kUnitBlocks + q;   // block within the window
                        const uint32_t wa = wv[2 * q], wb = wv[2 * q + 1];
                        const uint32_t sa8 = wa >> 8, sb8 = wb >> 8;
                        const uint32_t l0 = (wa & 0x000F000Fu) | 0x64006400u, l1 = (wb & 0x000F000Fu) | 0x64006400u;
                        const uint32_t l2 = (sa8 & 0x000F000Fu) | 0x64006400u, l3 = (sb8 & 0x000F000Fu) | 0x64006400u;
                        const uint32_t h0 = (wa & 0x00F000F0u) | 0x64006400u, h1 = (wb & 0x00F000F0u) | 0x64006400u;
                        const uint32_t h2 = (sa8 & 0x00F000F0u) | 0x64006400u, h3 = (sb8 & 0x00F000F0u) | 0x64006400u;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const int col = nt * 8 + g;
                            const uint4 X = col < p.B ? xs[(size_t)col * kXStride + 4 * j + t] : make_uint4(0u, 0u, 0u, 0u);
                            const float2 bz = *reinterpret_cast<const float2*>(bias + j * kMaxCols + nt * 8 + 2 * t);
                            float c[4] = {bz.x, bz.y, bz.x, bz.y};
                            persist::mma16816(c, l0, l1, l2, l3, X.x, X.y);
                            persist::mma16816(c, h0, h1, h2, h3, X.z, X.w);
                            if (first) {
                                acc0[nt][0] = fmaf(da[q], c[0], acc0[nt][0]);
                                acc0[nt][1] = fmaf(da[q], c[1], acc0[nt][1]);
                                acc0[nt][2] = fmaf(db[q], c[2], acc0[nt][2]);
                                acc0[nt][3] = fmaf(db[q], c[3], acc0[nt][3]);
                            } else {
                                acc1[nt][0] = fmaf(da[q], c[0], acc1[nt][0]);
                                acc1[nt][1] = fmaf(da[q], c[1], acc1[nt][1]);
                                acc1[nt][2] = fmaf(db[q], c[2], acc1[nt][2]);
                                acc1[nt][3] = fmaf(db[q], c[3], acc1[nt][3]);
                            }
                        }
                    }
                }
                __syncwarp();
                ++r.consumed;
                bring_issue(r, M, G, warp, lane);   // refill the slot just read
                u += n;
            }
        }
        // end of the group: finish the tiles this warp covered entirely, park the others
        __syncthreads();   // xs is free: part aliases it
        const int gt0 = G.T0 + kGroupTiles * gi;
        if (a < b) {
#pragma unroll
            for (int s2 = 0; s2 < 2; ++s2) {
                const int tl = s2 == 0 ? tl0 : tl1;
                if (s2 == 1 && tl1 == tl0) break;
                const float (&acc)[NT][4] = s2 == 0 ? acc0 : acc1;
                const bool owned = a <= tl * G.kwu && b >= (tl + 1) * G.kwu;
                if (owned) {
                    finish_tile<NT>(p, gt0 + tl, acc, kred, lane);
                } else {
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        part[((warp * 2 + s2) * NT + nt) * 32 + lane] =
                            make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
                }
            }
        }
        __syncthreads();
        // a shared tile is finished by the warp holding its last unit, summing in warp order
        if (a < b) {
            const int ts = tl0 * G.kwu;
            if (a > ts && b >= ts + G.kwu) {
                const int U = group_tiles(G, gi) * G.kwu;
                float s[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) s[nt][i] = 0.f;
                for (int w2 = 0; w2 <= warp; ++w2) {
                    const int a2 = persist::warp_unit<kW>(U, w2), b2 = persist::warp_unit<kW>(U, w2 + 1);
                    if (b2 <= a2 || b2 <= ts || a2 >= ts + G.kwu) continue;
                    const int sl = (a2 / G.kwu == tl0) ? 0 : 1;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const float4 v = part[((w2 * 2 + sl) * NT + nt) * 32 + lane];
                        s[nt][0] += v.x;
                        s[nt][1] += v.y;
                        s[nt][2] += v.z;
                        s[nt][3] += v.w;
                    }
                }
                finish_tile<NT>(p, gt0 + tl0, s, kred, lane);
            }
        }
    }
    if (p.epi == kEpiArgmax) {
        __syncthreads();
        if (tid < p.B) {
            const bool act = p.active == nullptr || p.active[tid] != 0;
            if (kred[tid] && act) atomicMax(p.keys + tid, kred[tid]);
        }
    }
    // after a wait ran out: let the copies in flight land (bounded) before leaving
    const unsigned long long t0 = persist::global_ns();
    while (r.consumed < r.issued) {
        const uint32_t mb = r.mbar + (r.consumed % kStages) * 8, parity = (r.consumed / kStages) & 1u;
        bool landed = persist::mbar_test(mb, parity);
        while (!landed && persist::global_ns() - t0 <= p.timeout_ns) landed = persist::mbar_test(mb, parity);
        if (!landed) break;
        ++r.consumed;
    }
}

// rs[b] = 1 / sqrt(mean_k x[b][k]^2 + eps): one CTA per column, fixed summation order.
__global__ void __launch_bounds__(256) rms_stats_kernel(const float* x, int cols, float eps, float* rs) {
    __shared__ float red[8];
    const int b = blockIdx.x, tid = threadIdx.x;
    pdl_wait();
    pdl_trigger();
    const float4* xb = reinterpret_cast<const float4*>(x + (size_t)b * cols);
    float ss = 0.f;
    for (int i = tid; i < cols / 4; i += 4 * 256) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = i + u * 256 < cols / 4 ? __ldcg(xb + i + u * 256) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < 4; ++u) ss += v[u].x * v[u].x + v[u].y * v[u].y + v[u].z * v[u].z + v[u].w * v[u].w;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    __syncthreads();
    if (tid == 0) {
        float t = 0.f;
        for (int w = 0; w < 8; ++w) t += red[w];
        rs[b] = 1.0f / sqrtf(t / (float)cols + eps);
    }
}

template <int NT>
cudaError_t run(bool launch, const BParams* p, int grid, cudaStream_t s, bool pdl) {
    if (!launch) {
        int dev = 0, optin = 0;
        cudaFuncAttributes fa = {};
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, gemv_batched_kernel<NT>);
        if (e == cudaSuccess && kSmem + fa.sharedSizeBytes > (size_t)optin) return cudaErrorInvalidConfiguration;
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gemv_batched_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
        return e;
    }
    return ql::launch(gemv_batched_kernel<NT>, dim3(grid), dim3(kT), kSmem, s, pdl, *p);
}

}  // namespace batched

bool batched_gemv_shape_ok(int nblk) {
    const int nst = nblk / batched::kUnitBlocks;
    return nblk % batched::kUnitBlocks == 0 && nst > 0 && (nst < batched::kWinUnits || nst % batched::kWinUnits == 0);
}

int batched_gemv_prepare() {
    static std::mutex mu;
    static std::set<int> done;
    int dev = 0;
    QL_TRY_CUDA(cudaGetDevice(&dev));
    std::lock_guard<std::mutex> lk(mu);
    if (done.count(dev)) return QL_OK;
    cudaError_t e = batched::run<1>(false, nullptr, 0, nullptr, false);
    if (e == cudaSuccess) e = batched::run<2>(false, nullptr, 0, nullptr, false);
    if (e == cudaSuccess) e = batched::run<3>(false, nullptr, 0, nullptr, false);
    if (e == cudaSuccess) e = batched::run<4>(false, nullptr, 0, nullptr, false);
    if (e != cudaSuccess) return cuda_error(e, "batched gemv: kernel attributes");
    done.insert(dev);
    return QL_OK;
}

int batched_gemv_launch(const StreamGemvArgs& a, cudaStream_t s, bool pdl) {
    QL_REQUIRE(a.M.stream && batched_gemv_shape_ok(a.M.nblk),
               "batched gemv: cols must be 128, 256, ..., 896 or a multiple of 1024");
    QL_REQUIRE(a.batch >= 1 && a.batch <= batched::kMaxCols, "batched gemv: batch must be in [1, 32]");
    QL_REQUIRE(a.rms ? (a.xf && a.norm_w && a.rs) : a.x16 != nullptr, "batched gemv: null input");
    QL_REQUIRE(a.y && a.sync, "batched gemv: null output");
    QL_REQUIRE(a.epilogue != kEpiArgmax || a.keys, "batched gemv: argmax needs keys");
    QL_REQUIRE((a.epilogue == QL_EPI_SILU_MUL) == (a.M.silu != 0), "batched gemv: SiLU*up needs a matrix packed for it");
    DevError* err = device_error_record();
    if (!err) return set_error(QL_ECUDA, "batched gemv: no device error record");
    if (int rc = batched_gemv_prepare()) return rc;
    batched::BParams p = {};
    p.M = a.M;
    p.B = a.batch;
    p.epi = a.epilogue;
    p.rms = a.rms;
    p.xf = a.xf;
    p.x16 = a.x16;
    p.norm_w = a.norm_w;
    p.eps = a.eps;
    p.y = a.y;
    if (a.rms) {   // the RMSNorm statistics of every column, once, for all CTAs
        const cudaError_t e0 = ql::launch(batched::rms_stats_kernel, dim3(a.batch), dim3(256), 0, s, pdl, a.xf,
                                          a.M.nblk * 32, a.eps, a.rs);
        if (e0 != cudaSuccess) return cuda_error(e0, "rms stats launch");
        p.rs_in = a.rs;
    }
    p.ld = a.ld;
    p.keys = a.keys;
    p.active = a.active;
    p.sync = a.sync;
    p.err = err;
    p.timeout_ns = 2000000000ull;
    const int nt = (a.batch + 7) / 8, grid = num_sms();
    cudaError_t e = nt == 1   ? batched::run<1>(true, &p, grid, s, pdl)
                    : nt == 2 ? batched::run<2>(true, &p, grid, s, pdl)
                    : nt == 3 ? batched::run<3>(true, &p, grid, s, pdl)
                              : batched::run<4>(true, &p, grid, s, pdl);
    if (e != cudaSuccess) return cuda_error(e, "batched gemv launch");
    return QL_OK;
}

}  // namespace ql
