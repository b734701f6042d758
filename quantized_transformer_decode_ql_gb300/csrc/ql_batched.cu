// Batched q4_0 GEMV (batch 3-32) over the tile stream layout: every weight byte is streamed
// once per call, whatever the batch.
//
// [IL] inferencelayer cuda_llm.rs, CudaQwen3::gemv (the q4_0 format, one GEMV per projection
// group) at the batch sizes where it becomes a skinny GEMM: each weight is used batch times, so
// the products go to the tensor cores (mma.sync m16n8k16, f16 in, f32 accumulate). The A
// fragment is the dequantised weight: the nibble expansion of the batch-1 kernel (1024 + q and
// 1024 + 16 q, exact) less its offset (q - 8 and 16 (q - 8), exact), times the block's f16 scale
// (one rounding to f16); a block's products then go straight into the f32 accumulator, so the
// dequantisation is paid once per weight for all batch columns.
//
// Why this shape (GB300): the activations of all batch columns for the full K (32 columns x
// 12288 x f16 = 768 KB for the down projection) do not fit in shared memory next to the weight
// ring, and re-reading the weights per column group multiplies the step's dominant traffic. So
// the GEMV is split over K: a CTA takes one K window of 1024 columns and one group of rows,
// stages that window of every batch column once, and streams the window's units of its tiles
// (at 1-3 tiles per CTA a row split alone would leave a window less than one unit per warp).
// The CTA writes f32 partial sums; a second kernel, over every SM, adds each output's windows
// in window order (deterministic) and applies the epilogue (a merge left to one CTA per row
// group made that CTA the launch's long tail). The weights arrive through the same per-warp
// ring of bulk copies (TMA) as the batch-1 kernel.
#include "ql_persist.cuh"

#include <atomic>
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
constexpr int kMaxCols = 32;                       // batch columns per call
constexpr int kXStride = kWinUnits * kUnitBlocks * 4 + 4;   // uint4 per staged column (+64 B)
constexpr size_t kRing = (size_t)kW * kStages * kSlotBytes;
constexpr size_t kXBytes = (size_t)kMaxCols * kXStride * 16;   // one window of every column
constexpr size_t kPartBytes = (size_t)kW * 2 * 4 * 32 * 16;    // [warp][slot][n-tile][lane] float4
constexpr size_t kXPart = kXBytes > kPartBytes ? kXBytes : kPartBytes;
constexpr size_t kSmem = kRing + kXPart;

struct BParams {
    PMat M;
    int B, epi;
    const __half* x16;     // f16 [B][cols] (RMSNorm'd inputs: written by rms_norm_kernel)
    void* y;
    int ld;
    unsigned long long* keys;
    const int32_t* active;
    unsigned int* sync;    // [4]: [2] is the abort flag of the bounded waits
    DevError* err;
    unsigned long long timeout_ns;
    float* part;           // [nwin][ntile * 16][kMaxCols] f32 partial sums of the K windows
    int ngr;               // row groups (grid = nwin * ngr)
    unsigned long long* trace;   // optional [grid][8] globaltimer stamps: 0 start, 1 past the wait,
                                 // 2 staged, 3 units done, 4 partials written, 5 end
};

// This CTA's K window and row group: CTA c = (window c % nwin, row group c / nwin).
struct Geo {
    int T0, T1, nst, kwu, nwin, w, rg;
};
__device__ __forceinline__ Geo geometry(const BParams& p) {
    Geo G;
    G.nst = p.M.nblk / kUnitBlocks;
    G.kwu = G.nst < kWinUnits ? G.nst : kWinUnits;
    G.nwin = G.nst / G.kwu;
    G.w = (int)blockIdx.x % G.nwin;
    G.rg = (int)blockIdx.x / G.nwin;
    G.T0 = (int)(((long long)G.rg * p.M.ntile) / p.ngr);
    G.T1 = (int)(((long long)(G.rg + 1) * p.M.ntile) / p.ngr);
    return G;
}

// Issue side of the ring: this warp's units [u, b) of the CTA's (tile, unit-of-window) list,
// tile-major; a copy never crosses a tile's run of kwu units.
struct BRing {
    int u, b;
    unsigned int issued, consumed;
    uint32_t base, mbar;
    int dead;
};
__device__ __forceinline__ void bring_issue(BRing& r, const PMat& M, const Geo& G, int lane) {
    if (r.u >= r.b || r.dead) return;
    const int tl = G.kwu == 8 ? r.u >> 3 : r.u / G.kwu, kk = r.u - tl * G.kwu;
    int n = r.b - r.u;
    n = n < kSlotUnits ? n : kSlotUnits;
    n = n < G.kwu - kk ? n : G.kwu - kk;
    if (lane == 0) {
        const int tile = G.T0 + tl, k = G.kwu * G.w + kk;
        const unsigned int slot = r.issued % kStages;
        const uint32_t mb = r.mbar + slot * 8, dst = r.base + slot * kSlotBytes;
        const uint32_t bytes = (uint32_t)(n * kUnitBytes);
        const uint8_t* src = M.stream + ((size_t)tile * G.nst + k) * kUnitBytes;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mb), "r"(bytes) : "memory");
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
                     ::"r"(dst), "l"(src), "r"(bytes), "r"(mb), "l"(l2_evict_first()) : "memory");
    }
    ++r.issued;
    r.u += n;
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

// Stage window w of every column: f16 pairs in the order a code word expands to (high ones
// pre-divided by 16, which is exact). Columns past the batch are never read.
__device__ void stage_window(const BParams& p, const Geo& G, int w, uint4* xs) {
    const int tid = threadIdx.x;
    const int nb = G.kwu * kUnitBlocks;        // blocks in the window
    const int cols = p.M.nblk * 32;
    const int j0 = w * nb;
    // the columns of the last 8-column tile past the batch are zero (read, never stored)
    const int pad = ((p.B + 7) & ~7) - p.B;
    for (int i = tid; i < pad * nb * 4; i += kT)
        xs[(size_t)(p.B + i / (nb * 4)) * kXStride + i % (nb * 4)] = make_uint4(0u, 0u, 0u, 0u);
    const int nitems = p.B * nb * 4;
    constexpr int kChunk = 4;   // items per thread whose loads are in flight together
    for (int base = 0; base < nitems; base += kChunk * kT) {
        uint2 ha[kChunk], hh[kChunk];
#pragma unroll
        for (int r = 0; r < kChunk; ++r) {
            const int item = base + r * kT + tid;
            if (item < nitems) {
                const int t = item & 3, cj = item >> 2, c = nb == 32 ? cj >> 5 : cj / nb, j = cj - c * nb;
                const size_t off = (size_t)c * cols + 32 * (j0 + j) + 4 * t;
                ha[r] = __ldcg(reinterpret_cast<const uint2*>(p.x16 + off));
                hh[r] = __ldcg(reinterpret_cast<const uint2*>(p.x16 + off + 16));
            }
        }
#pragma unroll
        for (int r = 0; r < kChunk; ++r) {
            const int item = base + r * kT + tid;
            if (item >= nitems) break;
            const int t = item & 3, cj = item >> 2, c = nb == 32 ? cj >> 5 : cj / nb, j = cj - c * nb;
            // elements 4t..4t+3 (ha) and 16+4t.. (hh): pairs (x0, x2), (x1, x3), (x16, x18)/16, (x17, x19)/16
            const float2 f0 = __half22float2(as_h2(ha[r].x)), f1 = __half22float2(as_h2(ha[r].y));
            const float2 f2 = __half22float2(as_h2(hh[r].x)), f3 = __half22float2(as_h2(hh[r].y));
            const __half2 p0 = __floats2half2_rn(f0.x, f1.x);
            const __half2 p1 = __floats2half2_rn(f0.y, f1.y);
            const __half2 p2 = __floats2half2_rn(f2.x * 0.0625f, f3.x * 0.0625f);
            const __half2 p3 = __floats2half2_rn(f2.y * 0.0625f, f3.y * 0.0625f);
            xs[(size_t)c * kXStride + 4 * j + t] = make_uint4(as_u32(p0), as_u32(p1), as_u32(p2), as_u32(p3));
        }
    }
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// Write this lane's fragment of a tile's partial sums for the CTA's window (rows g, g + 8 of
// the tile; columns 8 nt + 2t, +1).
template <int NT>
__device__ __forceinline__ void write_partial(const BParams& p, const Geo& G, int tile, const float (&acc)[NT][4],
                                              int lane) {
    const int g = lane >> 2, t = lane & 3;
    float* base = p.part + ((size_t)G.w * p.M.ntile + tile) * 16 * kMaxCols;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int c = nt * 8 + 2 * t;
        if (c < p.B) {
            base[g * kMaxCols + c] = acc[nt][0];
            base[(g + 8) * kMaxCols + c] = acc[nt][2];
        }
        if (c + 1 < p.B) {
            base[g * kMaxCols + c + 1] = acc[nt][1];
            base[(g + 8) * kMaxCols + c + 1] = acc[nt][3];
        }
    }
}

// The result: every output's window partials summed in window order, then the epilogue. An
// item is one output row and 8 columns (one 32-byte sector of a partial row per window);
// consecutive threads take consecutive rows, so the stores to y [column][row] coalesce. The
// loads of up to kMergeWin windows are in flight together. Grid-stride over the whole matrix.
constexpr int kMergeWin = 8, kMergeT = 256;
__global__ void __launch_bounds__(kMergeT) merge_kernel(const __grid_constant__ BParams p) {
    __shared__ unsigned long long kred[kMaxCols];
    if (threadIdx.x < kMaxCols) kred[threadIdx.x] = 0ull;
    pdl_wait();
    pdl_trigger();
    __syncthreads();
    const int nst = p.M.nblk / kUnitBlocks, kwu = nst < kWinUnits ? nst : kWinUnits, nwin = nst / kwu;
    const bool silu = p.epi == QL_EPI_SILU_MUL, resid = p.epi == QL_EPI_ADD_RESIDUAL;
    const int rpt = silu ? 8 : 16;                         // output rows per tile
    const int nrows = p.M.ntile * rpt, c8n = (p.B + 7) >> 3;
    const int lim = silu ? (p.M.rows >> 1) : p.M.rows;
    const size_t wstride = (size_t)p.M.ntile * 16 * (kMaxCols / 4);   // float4 per window
    const float4* part = reinterpret_cast<const float4*>(p.part);
    float* yf = static_cast<float*>(p.y);
    const long long nitems = (long long)nrows * c8n;
    for (long long i = blockIdx.x * (long long)kMergeT + threadIdx.x; i < nitems; i += (long long)gridDim.x * kMergeT) {
        // (no divisions: at most 4 column groups, 8 or 16 rows per tile)
        const int c8 = i < nrows ? 0 : i < 2ll * nrows ? 1 : i < 3ll * nrows ? 2 : 3;
        const int lr = (int)(i - (long long)c8 * nrows);
        const int tile = silu ? lr >> 3 : lr >> 4, r = lr - tile * rpt;
        const int row = tile * rpt + r;
        if (row >= lim) continue;
        const float4* q = part + ((size_t)tile * 16 + r) * (kMaxCols / 4) + 2 * c8;
        float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        float su[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        float res[8];   // the residual, loaded with the first windows
        if (resid) {
#pragma unroll
            for (int k = 0; k < 8; ++k) res[k] = 8 * c8 + k < p.B ? __ldcg(yf + (size_t)(8 * c8 + k) * p.ld + row) : 0.f;
        }
        // SiLU*up reads two rows per window: half as many windows per round
        const int wpr = silu ? kMergeWin / 2 : kMergeWin;
        for (int w0 = 0; w0 < nwin; w0 += wpr) {
            float4 v[kMergeWin][2];
#pragma unroll
            for (int k = 0; k < kMergeWin; ++k) {
                const int wk = silu ? w0 + (k >> 1) : w0 + k;
                if ((silu ? (k >> 1) : k) < wpr && wk < nwin) {
                    // SiLU*up: odd k is the up row (8 rows further in the tile)
                    const float4* qw = q + (size_t)wk * wstride + (silu && (k & 1) ? 8 * (kMaxCols / 4) : 0);
                    v[k][0] = __ldcg(qw);
                    v[k][1] = __ldcg(qw + 1);
                }
            }
#pragma unroll
            for (int k = 0; k < kMergeWin; ++k) {
                const int wk = silu ? w0 + (k >> 1) : w0 + k;
                if ((silu ? (k >> 1) : k) < wpr && wk < nwin) {
                    float* t = silu && (k & 1) ? su : s;
                    t[0] += v[k][0].x; t[1] += v[k][0].y; t[2] += v[k][0].z; t[3] += v[k][0].w;
                    t[4] += v[k][1].x; t[5] += v[k][1].y; t[6] += v[k][1].z; t[7] += v[k][1].w;
                }
            }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int c = 8 * c8 + k;
            if (c >= p.B) break;
            if (silu) {
                static_cast<__half*>(p.y)[(size_t)c * p.ld + row] = __float2half_rn(persist::silu(s[k]) * su[k]);
            } else if (resid) {
                yf[(size_t)c * p.ld + row] = res[k] + s[k];
            } else {
                yf[(size_t)c * p.ld + row] = s[k];
                if (p.epi == kEpiArgmax) atomicMax(kred + c, persist::argmax_key(s[k], row));
            }
        }
    }
    if (p.epi == kEpiArgmax) {
        __syncthreads();
        if (threadIdx.x < p.B) {
            const bool act = p.active == nullptr || p.active[threadIdx.x] != 0;
            if (kred[threadIdx.x] && act) atomicMax(p.keys + threadIdx.x, kred[threadIdx.x]);
        }
    }
}

template <int NT>
__global__ void __launch_bounds__(kT, 1) gemv_batched_kernel(const __grid_constant__ BParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ __align__(8) unsigned long long mbar[kW * kStages];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    uint4* xs = reinterpret_cast<uint4*>(smem + kRing);
    float4* part = reinterpret_cast<float4*>(smem + kRing);   // after the units: the shared tiles
    const PMat& M = p.M;
    const Geo G = geometry(p);
    unsigned long long* tr = p.trace ? p.trace + (size_t)blockIdx.x * persist::kTraceWords : nullptr;
    persist::stamp(tr, 0);
    const int U = (G.T1 - G.T0) * G.kwu;
    const int a = persist::warp_unit<kW>(U, warp), b = persist::warp_unit<kW>(U, warp + 1);

    if (lane == 0)
        for (int i = 0; i < kStages; ++i)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(
                             static_cast<uint32_t>(__cvta_generic_to_shared(&mbar[warp * kStages + i]))) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();
    BRing r;
    r.u = a;
    r.b = b;
    r.issued = r.consumed = 0;
    r.dead = 0;
    r.base = static_cast<uint32_t>(__cvta_generic_to_shared(smem)) + (uint32_t)(warp * kStages * kSlotBytes);
    r.mbar = static_cast<uint32_t>(__cvta_generic_to_shared(&mbar[warp * kStages]));
#pragma unroll 1
    for (int i = 0; i < kStages; ++i) bring_issue(r, M, G, lane);
    pdl_wait();
    pdl_trigger();
    persist::stamp(tr, 1);
    stage_window(p, G, G.w, xs);
    __syncthreads();
    persist::stamp(tr, 2);

    const int lm = lane >> 3, lrow = lane & 7;
    const uint32_t a_lo = (uint32_t)(((lm >> 1) * 16 + (lm & 1) * 8 + lrow) * 16);
    const uint4* xcol = xs + (size_t)g * kXStride + t;   // this lane's B fragments: column 8 nt + g
    const unsigned char* ring_g = smem + (size_t)warp * kStages * kSlotBytes;
    const int tl_first = a < b ? a / G.kwu : 0;
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;
    float first[NT][4];   // the warp's first tile, when it shares it with the previous warp
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) first[nt][i] = 0.f;
    bool first_parked = false, last_parked = false;
#pragma unroll 1
    for (int u = a; u < b;) {
        const int tl = G.kwu == 8 ? u >> 3 : u / G.kwu, kk = u - tl * G.kwu;
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
            const __half2 off_lo = as_h2(0x64086408u), off_hi = as_h2(0x64806480u);   // 1032, 1152
#pragma unroll
            for (int q = 0; q < kUnitBlocks; ++q) {
                const int j = (kk + i) * kUnitBlocks + q;   // block within the window
                // the scales of rows g and g + 8 for block q, in both halves of a half2
                const uint32_t sa = (q & 2) ? sca.y : sca.x, sb = (q & 2) ? scb.y : scb.x;
                const __half2 da = (q & 1) ? __high2half2(as_h2(sa)) : __low2half2(as_h2(sa));
                const __half2 db = (q & 1) ? __high2half2(as_h2(sb)) : __low2half2(as_h2(sb));
                const uint32_t wa = wv[2 * q], wb = wv[2 * q + 1];
                const uint32_t sa8 = wa >> 8, sb8 = wb >> 8;
                // (q - 8) d and 16 (q - 8) d (against x / 16) in the A fragment: rows g (a0, a2) and g + 8
                const uint32_t l0 = as_u32(__hmul2(__hsub2(as_h2((wa & 0x000F000Fu) | 0x64006400u), off_lo), da));
                const uint32_t l1 = as_u32(__hmul2(__hsub2(as_h2((wb & 0x000F000Fu) | 0x64006400u), off_lo), db));
                const uint32_t l2 = as_u32(__hmul2(__hsub2(as_h2((sa8 & 0x000F000Fu) | 0x64006400u), off_lo), da));
                const uint32_t l3 = as_u32(__hmul2(__hsub2(as_h2((sb8 & 0x000F000Fu) | 0x64006400u), off_lo), db));
                const uint32_t h0 = as_u32(__hmul2(__hsub2(as_h2((wa & 0x00F000F0u) | 0x64006400u), off_hi), da));
                const uint32_t h1 = as_u32(__hmul2(__hsub2(as_h2((wb & 0x00F000F0u) | 0x64006400u), off_hi), db));
                const uint32_t h2 = as_u32(__hmul2(__hsub2(as_h2((sa8 & 0x00F000F0u) | 0x64006400u), off_hi), da));
                const uint32_t h3 = as_u32(__hmul2(__hsub2(as_h2((sb8 & 0x00F000F0u) | 0x64006400u), off_hi), db));
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const uint4 X = xcol[(size_t)nt * 8 * kXStride + 4 * j];
                    persist::mma16816(acc[nt], l0, l1, l2, l3, X.x, X.y);
                    persist::mma16816(acc[nt], h0, h1, h2, h3, X.z, X.w);
                }
            }
        }
        __syncwarp();
        if (!r.dead) ++r.consumed;   // after a timeout the drain below still waits for this copy
        bring_issue(r, M, G, lane);   // refill the slot just read
        u += n;
        if (u == b || kk + n == G.kwu) {   // the end of this warp's part of the tile
            // end of this warp's part of tile tl: write it if the warp had all of the tile's
            // units of the window, else keep it for the reduction below (first or last tile)
            const int ts = tl * G.kwu;
            if (a <= ts && u == ts + G.kwu) {
                write_partial<NT>(p, G, G.T0 + tl, acc, lane);
            } else if (tl == tl_first && !first_parked) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) first[nt][i] = acc[nt][i];
                first_parked = true;
            } else {
                last_parked = true;   // the last tile's part stays in acc
                break;
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;
        }
    }
    persist::stamp(tr, 3);
    __syncthreads();   // xs is no longer read: part aliases it
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        part[((warp * 2 + 0) * NT + nt) * 32 + lane] =
            first_parked ? make_float4(first[nt][0], first[nt][1], first[nt][2], first[nt][3]) : make_float4(0.f, 0.f, 0.f, 0.f);
        part[((warp * 2 + 1) * NT + nt) * 32 + lane] =
            last_parked ? make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
    // a tile shared by warps is completed by the warp holding its last unit (its first tile),
    // summing the parts in warp order
    if (a < b) {
        const int ts = tl_first * G.kwu;
        if (a > ts && b >= ts + G.kwu) {
            float s2[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) s2[nt][i] = 0.f;
            for (int w2 = 0; w2 <= warp; ++w2) {
                const int a2 = persist::warp_unit<kW>(U, w2), b2 = persist::warp_unit<kW>(U, w2 + 1);
                if (b2 <= a2 || b2 <= ts || a2 >= ts + G.kwu) continue;
                const int sl = a2 >= ts ? 0 : 1;   // begun in this tile: parked as that warp's first
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float4 v = part[((w2 * 2 + sl) * NT + nt) * 32 + lane];
                    s2[nt][0] += v.x;
                    s2[nt][1] += v.y;
                    s2[nt][2] += v.z;
                    s2[nt][3] += v.w;
                }
            }
            write_partial<NT>(p, G, G.T0 + tl_first, s2, lane);
        }
    }
    __syncthreads();
    persist::stamp(tr, 4);
    persist::stamp(tr, 5);
    if (tr != nullptr && tid == 0) tr[6] = tr[7] = 0ull;
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

// RMSNorm of every column, once for all CTAs of the GEMV: xn[b] = f16(x[b] / rms(x[b]) * w) with
// rms = sqrt(mean_k x[b][k]^2 + eps); one CTA per column, fixed summation order.
constexpr int kNormT = 256;
__global__ void __launch_bounds__(kNormT) rms_norm_kernel(const float* x, int cols, float eps, const float* w,
                                                          __half* xn) {
    __shared__ float red[kNormT / 32];
    __shared__ float rs;
    const int b = blockIdx.x, tid = threadIdx.x;
    pdl_wait();
    pdl_trigger();
    const float4* xb = reinterpret_cast<const float4*>(x + (size_t)b * cols);
    float ss = 0.f;
    for (int i = tid; i < cols / 4; i += 4 * kNormT) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = i + u * kNormT < cols / 4 ? __ldcg(xb + i + u * kNormT) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < 4; ++u) ss += v[u].x * v[u].x + v[u].y * v[u].y + v[u].z * v[u].z + v[u].w * v[u].w;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    __syncthreads();
    if (tid == 0) {
        float t = 0.f;
        for (int k = 0; k < kNormT / 32; ++k) t += red[k];
        rs = rsqrtf(fmaf(t, 1.0f / (float)cols, eps));
    }
    __syncthreads();
    const float rr = rs;
    const float4* wv = reinterpret_cast<const float4*>(w);
    uint2* ob = reinterpret_cast<uint2*>(xn + (size_t)b * cols);
    for (int i = tid; i < cols / 4; i += 4 * kNormT) {   // a chunk's loads are all issued first
        float4 v[4], g[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (i + u * kNormT < cols / 4) {
                v[u] = __ldcg(xb + i + u * kNormT);
                g[u] = __ldg(wv + i + u * kNormT);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (i + u * kNormT < cols / 4) {
                const __half2 lo = __floats2half2_rn(v[u].x * rr * g[u].x, v[u].y * rr * g[u].y);
                const __half2 hi = __floats2half2_rn(v[u].z * rr * g[u].z, v[u].w * rr * g[u].w);
                ob[i + u * kNormT] = make_uint2(as_u32(lo), as_u32(hi));
            }
        }
    }
}

// ------------------------------------------------------------------ tcgen05 form
// The same split over K, with the products on the 5th-generation tensor cores: per row block of
// 8 tiles (128 rows, the MMA's M) and unit of the window, 16 dequantisation warps write the
// block's (q - 8) d into tensor memory (one thread per row: its 16-byte code runs expand, with
// LOP3 / HSUB2 / HMUL2, to the f16 values of the A operand, `tcgen05.st`), and one control warp
// issues `tcgen05.mma` (kind::f16, M = 128, N = 32 batch columns, K = 16) against the window's
// activations staged once in shared memory (the B operand, K-major core matrices), accumulating
// in f32 in tensor memory. The K order inside a 32-bit code word is the same permutation on both
// operands (the staged pairs of stage_window), so the sums are exact dot products. The codes
// stream in by bulk copies (one per tile per row block, 2 row blocks in flight); the
// accumulators of a row block are read back (`tcgen05.ld`) by 4 warps and written as the
// window's partial sums for merge_kernel. Every wait is bounded.
namespace tc {
constexpr int kDW = 16;                        // dequantisation warps, 4 per tensor-memory lane quarter
constexpr int kCtl = kDW;                      // the control warp (allocation, MMA issue)
constexpr int kThreads = (kDW + 1) * 32;
constexpr int kRB = 8;                         // tiles per row block: 128 rows
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kACol = 64;                 // A slots: kASlots x 64 columns from here; D: 2 x 32 below
constexpr int kASlots = 7;                     // unit g of the CTA (row block x window units) uses slot g % 7
constexpr size_t kCodesBytes = (size_t)kRB * kWinUnits * kUnitBytes;   // one row block's codes
constexpr size_t kBBytes = (size_t)kWinUnits * kUnitBlocks * 4 * 4 * 128;   // window x 32 columns, f16
constexpr size_t kSmem = 2 * kCodesBytes + kBBytes;
// MMA instruction descriptor: D f32, A and B f16, both K-major, N = 32, M = 128
constexpr uint32_t kIdesc = (1u << 4) | ((32u >> 3) << 17) | ((128u >> 4) << 24);
enum { kFull = 0, kFree = 2, kAFull = 4, kAFree = 4 + kASlots, kDFull = 4 + 2 * kASlots, kDFree = kDFull + 2,
       kDone = kDFree + 2, kBars = kDone + 1 };

__device__ __forceinline__ uint32_t su32(const void* q) { return static_cast<uint32_t>(__cvta_generic_to_shared(q)); }

// Wait for phase `parity` of an mbarrier, bounded; false (the CTA's abort flag set and the
// error recorded) when the bound runs out, or when another warp has aborted. abort_flag may be
// null (the final drain: the bound alone).
__device__ __forceinline__ bool tc_wait(uint32_t mb, uint32_t parity, const BParams& p, int* abort_flag, int where) {
    for (int spin = 0; spin < persist::kFastSpins; ++spin)
        if (persist::mbar_test(mb, parity)) return true;
    const unsigned long long t0 = persist::global_ns();
    for (unsigned int spin = 1;; ++spin) {
        if (persist::mbar_test(mb, parity)) return true;
        if ((spin & 63u) == 0) {
            if (abort_flag != nullptr && *reinterpret_cast<volatile int*>(abort_flag)) return false;
            if (persist::global_ns() - t0 > p.timeout_ns) break;
        }
    }
    if (abort_flag == nullptr || atomicExch(abort_flag, 1) == 0) {
        record_device_error(p.err, kErrGemvStage, blockIdx.x, where);
        atomicExch(p.sync + 2, 1u);
    }
    return false;
}

__device__ __forceinline__ void arrive(uint32_t mb) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mb) : "memory");
}

// Stage window w of every column as the B operand: chunk kc = 4 j + t (8 f16: the pairs of
// stage_window) of column c at ((kc * 4 + c / 8) * 8 + c % 8) * 16; columns past the batch zero.
// An item is (column c, block j, chunk t); the 8 columns of a group are consecutive lanes, so a
// warp's 16-byte stores fill whole 128-byte rows (no bank conflicts).
__device__ void stage_b(const BParams& p, const Geo& G, unsigned char* bsm, int nthreads) {
    const int tid = threadIdx.x;
    const int nb = G.kwu * kUnitBlocks, cols = p.M.nblk * 32, j0 = G.w * nb;
    const int ncg = (p.B + 7) >> 3;   // column groups holding batch columns
    uint4* b4 = reinterpret_cast<uint4*>(bsm);
    for (int i = tid; i < (4 - ncg) * 8 * nb * 4; i += nthreads) {   // groups past the batch
        const int cg = ncg + i / (8 * nb * 4), r = i % (8 * nb * 4);
        b4[((r >> 3) * 4 + cg) * 8 + (r & 7)] = make_uint4(0u, 0u, 0u, 0u);
    }
    const int nitems = ncg * 8 * nb * 4;
    constexpr int kChunk = 4;
    for (int base = 0; base < nitems; base += kChunk * nthreads) {
        uint2 ha[kChunk], hh[kChunk];
#pragma unroll
        for (int r = 0; r < kChunk; ++r) {
            const int item = base + r * nthreads + tid;
            const int cl = item & 7, t = (item >> 3) & 3, rest = item >> 5;
            const int cg0 = nb == 32 ? rest >> 5 : rest / nb, j = rest - cg0 * nb, c = cg0 * 8 + cl;
            if (item < nitems && c < p.B) {
                const size_t off = (size_t)c * cols + 32 * (j0 + j) + 4 * t;
                ha[r] = __ldcg(reinterpret_cast<const uint2*>(p.x16 + off));
                hh[r] = __ldcg(reinterpret_cast<const uint2*>(p.x16 + off + 16));
            } else {
                ha[r] = hh[r] = make_uint2(0u, 0u);
            }
        }
#pragma unroll
        for (int r = 0; r < kChunk; ++r) {
            const int item = base + r * nthreads + tid;
            if (item >= nitems) break;
            const int cl = item & 7, t = (item >> 3) & 3, rest = item >> 5;
            const int cg = nb == 32 ? rest >> 5 : rest / nb, j = rest - cg * nb;
            const float2 f0 = __half22float2(as_h2(ha[r].x)), f1 = __half22float2(as_h2(ha[r].y));
            const float2 f2 = __half22float2(as_h2(hh[r].x)), f3 = __half22float2(as_h2(hh[r].y));
            const __half2 p0 = __floats2half2_rn(f0.x, f1.x);
            const __half2 p1 = __floats2half2_rn(f0.y, f1.y);
            const __half2 p2 = __floats2half2_rn(f2.x * 0.0625f, f3.x * 0.0625f);
            const __half2 p3 = __floats2half2_rn(f2.y * 0.0625f, f3.y * 0.0625f);
            b4[((4 * j + t) * 4 + cg) * 8 + cl] = make_uint4(as_u32(p0), as_u32(p1), as_u32(p2), as_u32(p3));
        }
    }
}

// Bulk copy of tile i of row block rb (its units of the window, contiguous) into the row
// block's codes buffer; one lane. A tile past the row group only arrives.
__device__ __forceinline__ void issue_tile(const BParams& p, const Geo& G, unsigned char* codes, uint32_t bar, int rb,
                                           int i) {
    const int tl = rb * kRB + i, b = rb & 1;
    const uint32_t mb = bar + (kFull + b) * 8;
    if (tl >= G.T1 - G.T0) {
        arrive(mb);
        return;
    }
    const uint32_t bytes = (uint32_t)(G.kwu * kUnitBytes);
    const uint8_t* src = p.M.stream + ((size_t)(G.T0 + tl) * G.nst + (size_t)G.w * G.kwu) * kUnitBytes;
    const uint32_t dst = su32(codes + (size_t)b * kCodesBytes + (size_t)i * G.kwu * kUnitBytes);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mb), "r"(bytes) : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(mb), "l"(l2_evict_first()) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1) gemv_tc_kernel(const __grid_constant__ BParams p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ __align__(8) unsigned long long bars[kBars];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ int last_issued[2];   // per codes buffer: the last row block copied into it (-1: none)
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const Geo G = geometry(p);
    const int T = G.T1 - G.T0, nrb = (T + kRB - 1) / kRB, kwu = G.kwu;
    unsigned char* codes = smem;
    unsigned char* bsm = smem + 2 * kCodesBytes;
    const uint32_t bar = su32(bars);
    unsigned long long* tr = p.trace ? p.trace + (size_t)blockIdx.x * persist::kTraceWords : nullptr;
    persist::stamp(tr, 0);
    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar + (kFull + b) * 8), "r"(kRB) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar + (kFree + b) * 8), "r"(kDW) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar + (kDFull + b) * 8) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;" ::"r"(bar + (kDFree + b) * 8) : "memory");
            last_issued[b] = -1;
        }
        for (int a = 0; a < kASlots; ++a) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;" ::"r"(bar + (kAFull + a) * 8) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar + (kAFree + a) * 8) : "memory");
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar + kDone * 8) : "memory");
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kCtl) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&tmem_base)),
                     "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tb = tmem_base;
    int* abt = &abort_flag;

    // the first two row blocks' codes before the wait (the weights do not depend on the predecessor)
    if (warp < kRB && lane == 0) {
        for (int rb = 0; rb < 2 && rb < nrb; ++rb) {
            issue_tile(p, G, codes, bar, rb, warp);
            last_issued[rb] = rb;
        }
    }
    pdl_wait();
    pdl_trigger();
    persist::stamp(tr, 1);
    if (warp < kDW) stage_b(p, G, bsm, kDW * 32);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // B is read by the tensor cores
    __syncthreads();
    persist::stamp(tr, 2);

    if (warp < kDW) {
        const int q = warp & 3, sub = warp >> 2;
        const int nks = sub < kwu ? (kwu - sub + 3) / 4 : 0;   // units of the window this warp expands
        const int tr_ = 2 * q + (lane >> 4), rit = lane & 15;   // this thread's row: tile, row in tile
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const __half2 off_lo = as_h2(0x64086408u), off_hi = as_h2(0x64806480u);   // 1032, 1152
        auto epilogue = [&](int rb) {
            const int d = rb & 1;
            if (!tc_wait(bar + (kDFull + d) * 8, (uint32_t)(rb >> 1) & 1u, p, abt, 1000 + rb)) return false;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            uint32_t v[32];
            asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                         "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                         : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                           "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
                           "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]),
                           "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]),
                           "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
                         : "r"(tb + lane_base + 32u * (uint32_t)d) : "memory");
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) arrive(bar + (kDFree + d) * 8);
            const int tl = rb * kRB + tr_;
            if (tl < T) {
                float4* dst = reinterpret_cast<float4*>(p.part + (((size_t)G.w * p.M.ntile + G.T0 + tl) * 16 + rit) * kMaxCols);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    dst[c] = make_float4(__uint_as_float(v[4 * c]), __uint_as_float(v[4 * c + 1]),
                                         __uint_as_float(v[4 * c + 2]), __uint_as_float(v[4 * c + 3]));
            }
            return true;
        };
        bool ok = true;
        for (int rb = 0; rb < nrb && ok; ++rb) {
            const int b = rb & 1;
            // refill the other buffer with row block rb + 1 once every warp is done with rb - 1
            if (warp < kRB && rb >= 1 && rb + 1 < nrb) {
                if (lane == 0) {
                    ok = tc_wait(bar + (kFree + ((rb + 1) & 1)) * 8, (uint32_t)((rb - 1) >> 1) & 1u, p, abt, 2000 + rb);
                    if (ok) {
                        issue_tile(p, G, codes, bar, rb + 1, warp);
                        last_issued[(rb + 1) & 1] = rb + 1;
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
            }
            if (!tc_wait(bar + (kFull + b) * 8, (uint32_t)(rb >> 1) & 1u, p, abt, 3000 + rb)) {
                ok = false;
                break;
            }
            const unsigned char* cb = codes + (size_t)b * kCodesBytes;
            for (int k2 = 0; k2 < nks; ++k2) {
                const int kk = sub + 4 * k2, g = rb * kwu + kk, slot = g % kASlots, use = g / kASlots;
                if (use > 0 && !tc_wait(bar + (kAFree + slot) * 8, (uint32_t)(use - 1) & 1u, p, abt, 4000 + rb)) {
                    ok = false;
                    break;
                }
                const int tl = rb * kRB + tr_;
                const unsigned char* unit = cb + ((size_t)tr_ * kwu + kk) * kUnitBytes;
                const uint32_t ta = tb + lane_base + kACol + 64u * (uint32_t)slot;
#pragma unroll
                for (int half = 0; half < 2; ++half) {   // blocks 2 half, 2 half + 1: 32 columns
                    uint32_t v[32];
                    if (tl < T) {
                        const uint2 sc = *reinterpret_cast<const uint2*>(unit + 1024 + rit * 8);
                        const uint32_t sw = half ? sc.y : sc.x;
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int qb = 2 * half + e;
                            const uint4 cw = *reinterpret_cast<const uint4*>(unit + (qb * 16 + rit) * 16);
                            const __half2 d2 = e ? __high2half2(as_h2(sw)) : __low2half2(as_h2(sw));
                            const uint32_t ws[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                const uint32_t w = ws[t], w8 = w >> 8;
                                v[(e * 4 + t) * 4 + 0] = as_u32(__hmul2(__hsub2(as_h2((w & 0x000F000Fu) | 0x64006400u), off_lo), d2));
                                v[(e * 4 + t) * 4 + 1] = as_u32(__hmul2(__hsub2(as_h2((w8 & 0x000F000Fu) | 0x64006400u), off_lo), d2));
                                v[(e * 4 + t) * 4 + 2] = as_u32(__hmul2(__hsub2(as_h2((w & 0x00F000F0u) | 0x64006400u), off_hi), d2));
                                v[(e * 4 + t) * 4 + 3] = as_u32(__hmul2(__hsub2(as_h2((w8 & 0x00F000F0u) | 0x64006400u), off_hi), d2));
                            }
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = 0u;
                    }
                    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
                                 "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
                                 ::"r"(ta + 32u * (uint32_t)half), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]),
                                   "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]),
                                   "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
                                   "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]),
                                   "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31]) : "memory");
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                __syncwarp();
                if (lane == 0) arrive(bar + (kAFull + slot) * 8);
            }
            if (!ok) break;
            __syncwarp();
            if (lane == 0) arrive(bar + (kFree + b) * 8);   // this warp is done with the buffer
            if (sub == 3 && rb >= 1) ok = epilogue(rb - 1);
        }
        if (ok && sub == 3 && nrb > 0) epilogue(nrb - 1);
    } else if (lane == 0) {
        // the control warp's single issuing thread
        const uint32_t bbase = su32(bsm);
        for (int rb = 0; rb < nrb; ++rb) {
            const int d = rb & 1;
            if (rb >= 2 && !tc_wait(bar + (kDFree + d) * 8, (uint32_t)((rb - 2) >> 1) & 1u, p, abt, 5000 + rb)) break;
            bool ok = true;
            for (int kk = 0; kk < kwu && ok; ++kk) {
                const int g = rb * kwu + kk, s = g % kASlots, use = g / kASlots;
                if (!tc_wait(bar + (kAFull + s) * 8, (uint32_t)use & 1u, p, abt, 6000 + rb)) {
                    ok = false;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t baddr = bbase + (uint32_t)(kk * 16 + ks * 2) * 512u;
                    const unsigned long long desc = (unsigned long long)((baddr & 0x3FFFFu) >> 4) |
                                                    ((unsigned long long)(512u >> 4) << 16) |
                                                    ((unsigned long long)(128u >> 4) << 32) | (1ull << 46);
                    const uint32_t acc = (kk | ks) ? 1u : 0u;
                    asm volatile("{\n .reg .pred pa;\n setp.ne.u32 pa, %4, 0;\n"
                                 " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, pa;\n}"
                                 ::"r"(tb + 32u * (uint32_t)d), "r"(tb + kACol + 64u * (uint32_t)s + 8u * (uint32_t)ks),
                                   "l"(desc), "r"(kIdesc), "r"(acc) : "memory");
                }
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                             ::"r"(bar + (kAFree + s) * 8) : "memory");
            }
            if (!ok) break;
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                         ::"r"(bar + (kDFull + d) * 8) : "memory");
        }
        // every MMA issued has completed before the tensor memory is released
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                     ::"r"(bar + kDone * 8) : "memory");
        tc_wait(bar + kDone * 8, 0u, p, nullptr, 7000);
    }
    persist::stamp(tr, 3);
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    persist::stamp(tr, 4);
    if (warp == kCtl) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tb), "r"(kTmemCols) : "memory");
    }
    // copies still in flight (only after an abort): let them land before the CTA leaves (bounded)
    if (tid == 0) {
        for (int b = 0; b < 2; ++b)
            if (last_issued[b] >= 0)
                tc_wait(bar + (kFull + b) * 8, (uint32_t)(last_issued[b] >> 1) & 1u, p, nullptr, 8000);
    }
    persist::stamp(tr, 5);
    if (tr != nullptr && tid == 0) tr[6] = tr[7] = 0ull;
}
}  // namespace tc

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

// K windows and row groups of the split: grid = nwin * ngr <= SMs.
static void batched_split(int nblk, int ntile, int sms, int& nwin, int& ngr) {
    const int nst = nblk / batched::kUnitBlocks;
    const int kwu = nst < batched::kWinUnits ? nst : batched::kWinUnits;
    nwin = nst / kwu;
    ngr = sms / nwin;
    if (ngr > ntile) ngr = ntile;
    if (ngr < 1) ngr = 1;
}

// Workspace: the windows' partial sums.
size_t batched_gemv_workspace_bytes(int rows, int nblk, int silu) {
    const int ntile = silu ? (rows / 2 + 7) / 8 : (rows + 15) / 16;
    int nwin, ngr;
    batched_split(nblk, ntile, num_sms(), nwin, ngr);
    return (size_t)nwin * ntile * 16 * batched::kMaxCols * sizeof(float);
}

// The tensor-core form of batch 3-32 (process-wide): mma.sync by default (measured faster on the
// decode step), tcgen05 with ql_set_batched_gemv_form or QL_BATCHED_TC=1.
static std::atomic<int> g_form{-1};
static int batched_form() {
    int f = g_form.load();
    if (f < 0) {
        const char* e = std::getenv("QL_BATCHED_TC");
        f = (e != nullptr && std::atoi(e) != 0) ? QL_BATCHED_TCGEN05 : QL_BATCHED_MMA_SYNC;
        int expect = -1;
        g_form.compare_exchange_strong(expect, f);
        f = g_form.load();
    }
    return f;
}
static bool use_tc() { return batched_form() == QL_BATCHED_TCGEN05; }

int batched_gemv_prepare() {
    static std::mutex mu;
    static std::set<int> done;
    int dev = 0;
    QL_TRY_CUDA(cudaGetDevice(&dev));
    std::lock_guard<std::mutex> lk(mu);
    if (done.count(dev)) return QL_OK;
    {
        int optin = 0;
        cudaFuncAttributes fa = {};
        cudaError_t e0 = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e0 == cudaSuccess) e0 = cudaFuncGetAttributes(&fa, batched::tc::gemv_tc_kernel);
        if (e0 == cudaSuccess && batched::tc::kSmem + fa.sharedSizeBytes > (size_t)optin) e0 = cudaErrorInvalidConfiguration;
        if (e0 == cudaSuccess)
            e0 = cudaFuncSetAttribute(batched::tc::gemv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)batched::tc::kSmem);
        if (e0 != cudaSuccess) return cuda_error(e0, "batched gemv: tcgen05 kernel attributes");
    }
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
    QL_REQUIRE(a.rms ? (a.xf && a.norm_w && a.xn) : a.x16 != nullptr, "batched gemv: null input");
    QL_REQUIRE(a.y && a.sync && a.workspace, "batched gemv: null output or workspace");
    QL_REQUIRE(a.workspace_bytes >= batched_gemv_workspace_bytes(a.M.rows, a.M.nblk, a.M.silu),
               "batched gemv: workspace too small");
    QL_REQUIRE(a.epilogue != kEpiArgmax || a.keys, "batched gemv: argmax needs keys");
    QL_REQUIRE((a.epilogue == QL_EPI_SILU_MUL) == (a.M.silu != 0), "batched gemv: SiLU*up needs a matrix packed for it");
    DevError* err = device_error_record();
    if (!err) return set_error(QL_ECUDA, "batched gemv: no device error record");
    if (int rc = batched_gemv_prepare()) return rc;
    int nwin, ngr;
    batched_split(a.M.nblk, a.M.ntile, num_sms(), nwin, ngr);
    batched::BParams p = {};
    p.M = a.M;
    p.B = a.batch;
    p.epi = a.epilogue;
    p.x16 = a.rms ? a.xn : a.x16;
    p.y = a.y;
    p.ld = a.ld;
    p.keys = a.keys;
    p.active = a.active;
    p.sync = a.sync;
    p.err = err;
    p.timeout_ns = 2000000000ull;
    p.part = static_cast<float*>(a.workspace);
    p.ngr = ngr;
    p.trace = a.trace;
    if (a.rms) {   // the RMSNorm'd activations of every column, once, for all CTAs
        const cudaError_t e0 = ql::launch(batched::rms_norm_kernel, dim3(a.batch), dim3(batched::kNormT), 0, s, pdl,
                                          a.xf, a.M.nblk * 32, a.eps, a.norm_w, a.xn);
        if (e0 != cudaSuccess) return cuda_error(e0, "rms norm launch");
    }
    const int nt = (a.batch + 7) / 8, grid = nwin * ngr;
    cudaError_t e;
    if (use_tc())
        e = ql::launch(batched::tc::gemv_tc_kernel, dim3(grid), dim3(batched::tc::kThreads), batched::tc::kSmem, s,
                       pdl, p);
    else
        e = nt == 1   ? batched::run<1>(true, &p, grid, s, pdl)
            : nt == 2 ? batched::run<2>(true, &p, grid, s, pdl)
            : nt == 3 ? batched::run<3>(true, &p, grid, s, pdl)
                      : batched::run<4>(true, &p, grid, s, pdl);
    if (e != cudaSuccess) return cuda_error(e, "batched gemv launch");
    // the windows added up and the epilogue, over every SM
    e = ql::launch(batched::merge_kernel, dim3(2 * num_sms()), dim3(batched::kMergeT), 0, s, pdl, p);
    if (e != cudaSuccess) return cuda_error(e, "batched gemv merge launch");
    return QL_OK;
}

}  // namespace ql

extern "C" int ql_set_batched_gemv_form(int form) {
    using namespace ql;
    QL_REQUIRE(form == QL_BATCHED_MMA_SYNC || form == QL_BATCHED_TCGEN05, "ql_set_batched_gemv_form: unknown form");
    const int prev = batched_form();
    g_form.store(form);
    return prev;
}
