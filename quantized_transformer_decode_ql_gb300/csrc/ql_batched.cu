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
#include "ql_batched.h"
#include "ql_persist.cuh"

#include <cuda.h>   // CUtensorMap and its enums (the encoder is taken from the driver at run time)

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
    float* part;           // [nwin][kMaxCols][ntile * 16] f32 partial sums of the K windows (per
                           // window and batch column, the rows in order: warp loads of 32
                           // consecutive rows of a column are one 128-byte line)
    int ngr;               // row groups (grid = nwin * ngr)
    int* tickets;          // tcgen05 form: [ngr][maxrb] window counts per row block, zero between calls
    int maxrb;             // row blocks (8 tiles) of the largest row group
    int kernel_merge;      // tcgen05 form: 1 = merge the K windows in the kernel (tickets), 0 = merge_kernel
    CUtensorMap tmap;      // tcgen05 form: the stream as [tile][unit][144 x 8 bytes], boxes of 8 tiles x 1 unit
    // RMSNorm folded into the merges (mma.sync form, decode step): a consumer GEMV stages x16 =
    // f16(x w) of its un-normalised input, and its merge multiplies the window sums of column c by
    // rsqrt(sum_i x_c[i]^2 / cols + eps), from ssq_in ([cols / 32][kMaxCols] sums over 32-row
    // chunks). A producer (residual epilogue) writes, besides the new x, xn_out = f16(x w_next)
    // ([B][rows]) and those chunk sums of the new x into ssq_out.
    const float* ssq_in;
    float* ssq_out;
    const float* w_next;
    __half* xn_out;
    float eps;
    unsigned long long* trace;   // optional [grid][8] globaltimer stamps: 0 start, 1 past the wait,
                                 // 2 staged, 3 units done, 4 partials written, 5 end
    unsigned long long* mtrace;  // merge_kernel's, optional [grid][kMergeTraceWords]: 0 start, 1 past
                                 // the wait, 2 items done, 3 end
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
// the tile; columns 8 nt + 2t, +1). Each store instruction writes 8 consecutive rows of 4
// columns: four 32-byte sectors.
template <int NT>
__device__ __forceinline__ void write_partial(const BParams& p, const Geo& G, int tile, const float (&acc)[NT][4],
                                              int lane) {
    const int g = lane >> 2, t = lane & 3;
    const int R = p.M.ntile * 16;   // (32 R is far below 2^31 for every supported shape)
    float* base = p.part + (size_t)G.w * kMaxCols * R + tile * 16 + g;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int c = nt * 8 + 2 * t;
        if (c < p.B) {
            base[c * R] = acc[nt][0];
            base[c * R + 8] = acc[nt][2];
        }
        if (c + 1 < p.B) {
            base[(c + 1) * R] = acc[nt][1];
            base[(c + 1) * R + 8] = acc[nt][3];
        }
    }
}

// The result: every output's window partials summed in window order, then the epilogue. An
// item is one output row and CG columns; consecutive threads take consecutive rows, so that
// both the partial loads (per window and column, a warp reads 32 consecutive rows: one line)
// and the stores to y [column][row] coalesce. The loads of up to 64 / CG windows (SiLU*up: half
// as many, two rows each) are in flight together: CG = 4 when a matrix has more than 8 K
// windows, so that the down projection's 12 windows take one round. One CTA of 512 threads per
// SM; the items go out warp by warp over the CTAs first (the 32 items of a warp are 32
// consecutive rows), so that a small matrix still spreads over every SM, and at batch 32 the
// gate|up merge is one round.
constexpr int kMergeT = 512;
template <int CG>
__global__ void __launch_bounds__(kMergeT, 1) merge_kernel(const __grid_constant__ BParams p) {
    constexpr int kWin = 64 / CG;        // windows per round of loads
    constexpr int kSl = 8;               // RMSNorm factor: chunk slices per column (threads < 256)
    __shared__ unsigned long long kred[kMaxCols];
    __shared__ float nred[kSl][kMaxCols];
    __shared__ float nf[kMaxCols];   // the RMSNorm factor per column (consumer form)
    unsigned long long* mt = p.mtrace ? p.mtrace + (size_t)blockIdx.x * kMergeTraceWords : nullptr;
    persist::stamp(mt, 0);
    if (threadIdx.x < kMaxCols) kred[threadIdx.x] = 0ull;
    if (p.ssq_in != nullptr) {
        // before the wait: the producer's merge that wrote the sums ran two launches back. Per
        // column, chunk slices summed in a fixed order (thread = column + 32 slice), then the slices
        if (threadIdx.x < kSl * kMaxCols) {
            const int c = threadIdx.x % kMaxCols, sl = threadIdx.x / kMaxCols, nch = p.M.nblk;
            float a = 0.f;
            for (int j = sl; j < nch; j += kSl) a += __ldcg(p.ssq_in + (size_t)j * kMaxCols + c);
            nred[sl][c] = a;
        }
        __syncthreads();
        if (threadIdx.x < kMaxCols) {
            float t = 0.f;
#pragma unroll
            for (int q = 0; q < kSl; ++q) t += nred[q][threadIdx.x];
            nf[threadIdx.x] = rsqrtf(fmaf(t, 1.0f / (float)(p.M.nblk * 32), p.eps));
        }
    }
    pdl_wait();
    pdl_trigger();
    persist::stamp(mt, 1);
    __syncthreads();
    const int nst = p.M.nblk / kUnitBlocks, kwu = nst < kWinUnits ? nst : kWinUnits, nwin = nst / kwu;
    const bool silu = p.epi == QL_EPI_SILU_MUL, resid = p.epi == QL_EPI_ADD_RESIDUAL;
    const int rpt = silu ? 8 : 16;                         // output rows per tile
    const int nrows = p.M.ntile * rpt, ncg = (p.B + CG - 1) / CG;
    const int lim = silu ? (p.M.rows >> 1) : p.M.rows;
    const size_t R = (size_t)p.M.ntile * 16;           // partial rows per window and column
    float* yf = static_cast<float*>(p.y);
    const long long nitems = (long long)nrows * ncg;
    const long long i0 = ((long long)(threadIdx.x >> 5) * gridDim.x + blockIdx.x) * 32 + (threadIdx.x & 31);
    for (long long i = i0; i < nitems; i += (long long)gridDim.x * kMergeT) {
        int cg = 0;   // (no division: at most 8 column groups)
        long long li = i;
        while (li >= nrows) {
            li -= nrows;
            ++cg;
        }
        const int lr = (int)li;
        const int tile = silu ? lr >> 3 : lr >> 4, r = lr - tile * rpt;
        const int row = tile * rpt + r;
        if (row >= lim) continue;
        const int c0 = CG * cg;
        const int nc = p.B - c0 < CG ? p.B - c0 : CG;   // columns of this group in the batch
        // the partial row of column c0 in window 0 (SiLU*up: the gate row; the up row is 8 further)
        const float* q = p.part + (size_t)c0 * R + (size_t)tile * 16 + r;
        float s[CG], su[CG], res[CG];   // res: the residual, loaded with the first windows
#pragma unroll
        for (int k = 0; k < CG; ++k) s[k] = su[k] = 0.f;
        if (resid) {
#pragma unroll
            for (int k = 0; k < CG; ++k) res[k] = k < nc ? __ldcg(yf + (size_t)(c0 + k) * p.ld + row) : 0.f;
        }
        const int wpr = silu ? kWin / 2 : kWin;
        for (int w0 = 0; w0 < nwin; w0 += wpr) {
            float v[kWin][CG];
#pragma unroll
            for (int k = 0; k < kWin; ++k) {
                const int wk = silu ? w0 + (k >> 1) : w0 + k;
                if ((silu ? (k >> 1) : k) < wpr && wk < nwin) {
                    // SiLU*up: odd k is the up row (8 rows further in the tile)
                    const float* qw = q + (size_t)wk * kMaxCols * R + (silu && (k & 1) ? 8 : 0);
#pragma unroll
                    for (int j = 0; j < CG; ++j) v[k][j] = j < nc ? __ldcg(qw + (size_t)j * R) : 0.f;
                }
            }
#pragma unroll
            for (int k = 0; k < kWin; ++k) {
                const int wk = silu ? w0 + (k >> 1) : w0 + k;
                if ((silu ? (k >> 1) : k) < wpr && wk < nwin) {
                    float* t = silu && (k & 1) ? su : s;
#pragma unroll
                    for (int j = 0; j < CG; ++j) t[j] += v[k][j];
                }
            }
        }
        if (p.ssq_in != nullptr) {
#pragma unroll
            for (int k = 0; k < CG; ++k) {
                const float f = k < nc ? nf[c0 + k] : 0.f;
                s[k] *= f;
                su[k] *= f;
            }
        }
        if (resid && p.ssq_out != nullptr) {
            // the new x, f16(x w_next) for the next GEMV, and the 32-row chunk sums of x^2 (the
            // warp's 32 lanes hold 32 consecutive rows of one column group: a fixed shuffle tree)
            float sq[CG];
            const float wn = __ldg(p.w_next + row);
#pragma unroll
            for (int k = 0; k < CG; ++k) {
                const int c = c0 + k;
                float v = 0.f;
                if (k < nc) {
                    v = res[k] + s[k];
                    yf[(size_t)c * p.ld + row] = v;
                    p.xn_out[(size_t)c * p.M.rows + row] = __float2half_rn(v * wn);
                }
                sq[k] = v * v;
            }
#pragma unroll
            for (int k = 0; k < CG; ++k)
#pragma unroll
                for (int o = 16; o; o >>= 1) sq[k] += __shfl_xor_sync(0xffffffffu, sq[k], o);
            if ((threadIdx.x & 31) == 0) {
#pragma unroll
                for (int k = 0; k < CG; ++k)
                    if (k < nc) p.ssq_out[(size_t)(row >> 5) * kMaxCols + c0 + k] = sq[k];
            }
            continue;
        }
#pragma unroll
        for (int k = 0; k < CG; ++k) {
            const int c = c0 + k;
            if (k >= nc) break;
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
    if (mt != nullptr) {   // (the condition is the same for every thread of the CTA)
        __syncthreads();
        persist::stamp(mt, 2);
    }
    if (p.epi == kEpiArgmax) {
        __syncthreads();
        if (threadIdx.x < p.B) {
            const bool act = p.active == nullptr || p.active[threadIdx.x] != 0;
            if (kred[threadIdx.x] && act) atomicMax(p.keys + threadIdx.x, kred[threadIdx.x]);
        }
    }
    persist::stamp(mt, 3);
}

// the merge's launch: 4-column items above 8 K windows (see merge_kernel)
static cudaError_t launch_merge(const BParams& p, int nwin, cudaStream_t s, bool pdl) {
    if (nwin > 8) return ql::launch(merge_kernel<4>, dim3(num_sms()), dim3(kMergeT), 0, s, pdl, p);
    return ql::launch(merge_kernel<8>, dim3(num_sms()), dim3(kMergeT), 0, s, pdl, p);
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
    // one ring slot before the wait, the rest once the window's activation loads are out: in the
    // step a CTA often starts only as the merge before it ends, and staging loads queued behind
    // both slots' copies (E32 6382 vs 6325 tokens/s with both slots first, 6280 with none)
    bring_issue(r, M, G, lane);
    pdl_wait();
    pdl_trigger();
    persist::stamp(tr, 1);
    stage_window(p, G, G.w, xs);
#pragma unroll 1
    for (int i = 1; i < kStages; ++i) bring_issue(r, M, G, lane);
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
// The same split over K, with the products on the 5th-generation tensor cores and every stage
// of the work in its own warps, joined by mbarriers:
//  * a producer lane streams the codes into a ring of kS shared-memory stages, one stage = one
//    unit (128 columns) of every tile of a row block (8 tiles = 128 rows, the MMA's M): one
//    tensor-map copy of 8 tiles x 1 unit (single-tile copies for a row group's last, partial
//    row block), completing on the stage's mbarrier;
//  * 16 dequantisation warps in 4 groups (one warp per tensor-memory lane quarter each: the
//    warp of quarter q handles rows 32q..32q+31, tiles 2q and 2q+1 of the row block) take
//    groups of kPair units in turn: each thread expands its row's codes into (q - 8) d in f16
//    (LOP3 / HSUB2 / HMUL2, the K order of the staged activations) and stores them into one of
//    kA rotating A slots of tensor memory (`tcgen05.st`);
//  * one lane issues `tcgen05.mma` (kind::f16, M = 128, N = 32 batch columns, K = 16, A in
//    tensor memory, B = the window's activations staged once in shared memory as K-major core
//    matrices) into one of two f32 accumulators, and commits each group of units and each
//    finished row block to mbarriers;
//  * 4 epilogue warps read a finished row block's accumulator (`tcgen05.ld`) and write it as the
//    window's partial sums; merge_kernel adds the windows in window order, or (selectable) the
//    CTA that takes a row block's last ticket does (results do not depend on which CTA merges).
// Measured on GB300: one M128 N32 K16 MMA occupies the tensor core ~28 ns whatever N up to 64,
// ~35 ns while other warps store into tensor memory, so at N = 32 the products alone take about
// as long as streaming the weights; with the waits, fences and commits around each group the
// form runs behind the mma.sync form on the batch-32 step.
// Every wait is bounded; after a timeout the CTA records the error, stops, lets its copies in
// flight land and frees its tensor memory.
namespace tc {
constexpr int kDW = 16;                        // dequantisation warps, 4 per tensor-memory lane quarter
constexpr int kMmaWarp = kDW;                  // tensor-memory allocation; lane 0 issues the MMAs
constexpr int kProdWarp = kDW + 1;             // lane 0 issues the bulk copies
constexpr int kEpiWarp0 = kDW + 2;             // 4 epilogue warps (quarter = warp & 3)
constexpr int kWarps = kDW + 6, kThreads = kWarps * 32;
constexpr int kRB = 8;                         // tiles per row block: 128 rows
constexpr int kStageBytes = kRB * kUnitBytes;  // one unit of each tile of a row block
constexpr int kS = 16;                         // shared-memory stages
constexpr uint32_t kTmemCols = 512;
constexpr int kAcc = 1;                        // accumulators per set (32 columns each)
constexpr uint32_t kDCols = 32u * kAcc;        // one set
constexpr uint32_t kACol = 2 * kDCols;         // A slots after the two sets
constexpr int kPair = 2;                       // units of a row block per A slot (one MMA group)
constexpr int kA = (int)((kTmemCols - kACol) / (64 * kPair));   // A slots of kPair x 64 columns
constexpr size_t kBBytes = (size_t)kWinUnits * kUnitBlocks * 4 * 4 * 128;   // window x 32 columns, f16
constexpr size_t kSmem = (size_t)kS * kStageBytes + kBBytes;
// MMA instruction descriptor: D f32, A and B f16, both K-major, N = 32, M = 128
constexpr uint32_t kIdesc = (1u << 4) | ((32u >> 3) << 17) | ((128u >> 4) << 24);
constexpr int kGroups = kDW / 4;                // dequantisation groups (one warp per lane quarter each)
// Barriers. A waiter on phase k of an mbarrier must know that phase k - 1 has completed (a parity
// test cannot tell phase k - 1 from k + 1), so every barrier has one waiter role that takes its
// phases in order: the producer SFree, the group of a slot's stages SFull (stage s and s + kS
// always fall to the same group), the MMA lane AFull and DFree, the epilogue DFull, and each
// group its own AFreeG, which the MMA lane commits in that group's order of unit groups.
enum { kSFull = 0, kSFree = kS, kAFull = 2 * kS, kAFreeG = 2 * kS + kA, kDFull = 2 * kS + kA + kGroups,
       kDFree = kDFull + 2, kDone = kDFree + 2, kBars = kDone + 1 };
static_assert(kS % (2 * kGroups) == 0, "a slot's stages must fall to one group");
constexpr int kEpiBarrier = 1;                 // named barrier of the 4 epilogue warps

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

// tc_wait by every lane of a warp, with one answer for the warp (its collective tcgen05
// instructions that follow need every lane or none): false if any lane's wait failed.
__device__ __forceinline__ bool warp_wait(uint32_t mb, uint32_t parity, const BParams& p, int* abort_flag, int where) {
    const bool ok = tc_wait(mb, parity, p, abort_flag, where);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void arrive(uint32_t mb) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mb) : "memory");
}

// 16 consecutive 32-bit columns of this warp's 32 tensor-memory lanes, waited for.
__device__ __forceinline__ void tmem_ld16(uint32_t addr, uint32_t (&v)[16]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                   "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
                 : "r"(addr) : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void epi_sync() {
    asm volatile("bar.sync %0, %1;" ::"n"(kEpiBarrier), "n"(4 * 32) : "memory");
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

// Bulk copies of stage s (row block s / kwu, unit s % kwu of the window: that unit of each of
// the row block's tiles) into its shared-memory slot; one lane. Tiles past the row group are
// not copied (their rows are never written out).
__device__ __forceinline__ void issue_stage(const BParams& p, const Geo& G, unsigned char* ring, uint32_t bar, int rb,
                                            int kk, int slot, unsigned long long pol) {
    const int T = G.T1 - G.T0;
    const int nt = T - rb * kRB < kRB ? T - rb * kRB : kRB;
    const uint32_t mb = bar + (kSFull + slot) * 8;
    // the slot's previous contents were read through the generic proxy; the copy below writes it
    // through the async proxy
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mb), "r"((uint32_t)(nt * kUnitBytes))
                 : "memory");
    if (nt == kRB) {   // a whole row block: one tensor copy of 8 tiles x 1 unit
        asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
                     " [%0], [%1, {%2, %3, %4}], [%5], %6;"
                     ::"r"(su32(ring + (size_t)slot * kStageBytes)), "l"(reinterpret_cast<uint64_t>(&p.tmap)), "r"(0),
                       "r"(G.w * G.kwu + kk), "r"(G.T0 + rb * kRB), "r"(mb), "l"(pol) : "memory");
        return;
    }
    for (int i = 0; i < nt; ++i) {
        const uint8_t* src = p.M.stream + ((size_t)(G.T0 + rb * kRB + i) * G.nst + (size_t)G.w * G.kwu + kk) * kUnitBytes;
        const uint32_t dst = su32(ring + (size_t)slot * kStageBytes + (size_t)i * kUnitBytes);
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
                     ::"r"(dst), "l"(src), "r"((uint32_t)kUnitBytes), "r"(mb), "l"(pol) : "memory");
    }
}

// The merge of row block rb (tiles T0 + 8 rb ..) by the 4 epilogue warps: every output's window
// partials added in window order, then the epilogue. Thread e takes row e % 16 of each tile
// and columns 4 (e / 16) ..; per window and column a half warp reads 16 consecutive rows (64
// contiguous bytes). SiLU*up: the threads holding a gate row (row of the tile < 8) also read its
// up row 8 further; the others idle. Every epilogue thread runs the whole function, so that the
// argmax reduction can shuffle over full warps.
template <bool SILU>
__device__ __noinline__ void merge_rb(const BParams& p, const Geo& G, int rb, int e) {
    const bool resid = p.epi == QL_EPI_ADD_RESIDUAL, amax = p.epi == kEpiArgmax;
    const int T = G.T1 - G.T0, ntl = T - rb * kRB < kRB ? T - rb * kRB : kRB;
    const int rit = e & 15, c4 = e >> 4;                // row of the tile, column group
    const int lim = SILU ? (p.M.rows >> 1) : p.M.rows;
    const size_t R = (size_t)p.M.ntile * 16;           // partial rows per window and column
    const float* base = p.part + (size_t)4 * c4 * R + (size_t)(G.T0 + rb * kRB) * 16 + rit;
    float* yf = static_cast<float*>(p.y);
    constexpr int kJ = 4;                               // tiles per round
    for (int j0 = 0; j0 < kRB; j0 += kJ) {
        float4 sg[kJ], su[kJ];
#pragma unroll
        for (int j = 0; j < kJ; ++j) sg[j] = su[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        const bool lanes = !SILU || rit < 8;
        for (int w = 0; w < G.nwin; ++w) {
            float4 vg[kJ], vu[kJ];
#pragma unroll
            for (int j = 0; j < kJ; ++j) {
                if (lanes && j0 + j < ntl) {
                    const float* q = base + (size_t)w * kMaxCols * R + (size_t)(j0 + j) * 16;
                    vg[j] = make_float4(__ldcg(q), __ldcg(q + R), __ldcg(q + 2 * R), __ldcg(q + 3 * R));
                    if (SILU)   // row + 8 of the tile
                        vu[j] = make_float4(__ldcg(q + 8), __ldcg(q + R + 8), __ldcg(q + 2 * R + 8), __ldcg(q + 3 * R + 8));
                }
            }
#pragma unroll
            for (int j = 0; j < kJ; ++j) {
                if (lanes && j0 + j < ntl) {
                    sg[j].x += vg[j].x; sg[j].y += vg[j].y; sg[j].z += vg[j].z; sg[j].w += vg[j].w;
                    if (SILU) { su[j].x += vu[j].x; su[j].y += vu[j].y; su[j].z += vu[j].z; su[j].w += vu[j].w; }
                }
            }
        }
#pragma unroll
        for (int j = 0; j < kJ; ++j) {
            const int tile = G.T0 + rb * kRB + j0 + j;
            const int row = SILU ? tile * 8 + rit : tile * 16 + rit;
            const bool valid = lanes && j0 + j < ntl && row < lim;
            const float sv[4] = {sg[j].x, sg[j].y, sg[j].z, sg[j].w};
            const float uv[4] = {su[j].x, su[j].y, su[j].z, su[j].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int c = 4 * c4 + k;
                if (valid && c < p.B) {
                    if (SILU) {
                        static_cast<__half*>(p.y)[(size_t)c * p.ld + row] = __float2half_rn(persist::silu(sv[k]) * uv[k]);
                    } else if (resid) {
                        float* yp = yf + (size_t)c * p.ld + row;
                        *yp = __ldcg(yp) + sv[k];
                    } else {
                        yf[(size_t)c * p.ld + row] = sv[k];
                    }
                }
                if (!SILU && amax) {
                    // per column: the largest key over the lanes holding it (a half warp, e / 16
                    // equal), then one atomic per half warp and column
                    unsigned long long key = valid && c < p.B ? persist::argmax_key(sv[k], row) : 0ull;
#pragma unroll
                    for (int o = 1; o < 16; o <<= 1) {
                        const unsigned long long ok = __shfl_xor_sync(0xffffffffu, key, o);
                        key = ok > key ? ok : key;
                    }
                    const bool act = c < p.B && (p.active == nullptr || p.active[c] != 0);
                    if (act && key != 0ull && (threadIdx.x & 15) == 0) atomicMax(p.keys + c, key);
                }
            }
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1) gemv_tc_kernel(const __grid_constant__ BParams p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ __align__(8) unsigned long long bars[kBars];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ int merge_flag, epi_stop;
    __shared__ int issued_stages;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const Geo G = geometry(p);
    const int T = G.T1 - G.T0, nrb = (T + kRB - 1) / kRB, kwu = G.kwu, nstage = nrb * kwu;
    // units per A-slot group: kPair, or 1 when kwu is odd (then group g is stage g, and stages s and
    // s + kS still fall to the same dequantisation group)
    const int ps = (kwu % kPair) == 0 ? kPair : 1;
    const int npr = kwu / ps, npair = nrb * npr;
    unsigned char* ring = smem;
    unsigned char* bsm = smem + (size_t)kS * kStageBytes;
    const uint32_t bar = su32(bars);
    unsigned long long* tr = p.trace ? p.trace + (size_t)blockIdx.x * persist::kTraceWords : nullptr;
    persist::stamp(tr, 0);
    if (tid == 0) {
        for (int i = 0; i < kS; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar + (kSFull + i) * 8) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;" ::"r"(bar + (kSFree + i) * 8) : "memory");
        }
        for (int a = 0; a < kA; ++a)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;" ::"r"(bar + (kAFull + a) * 8) : "memory");
        for (int j = 0; j < kGroups; ++j)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar + (kAFreeG + j) * 8) : "memory");
        for (int d = 0; d < 2; ++d) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar + (kDFull + d) * 8) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;" ::"r"(bar + (kDFree + d) * 8) : "memory");
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar + kDone * 8) : "memory");
        abort_flag = 0;
        issued_stages = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&tmem_base)),
                     "r"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tb = tmem_base;
    int* abt = &abort_flag;

    // the first stages' codes before the wait (the weights do not depend on the predecessor);
    // (prb, pkk) is the row block and unit of stage `issued`
    int issued = 0, prb = 0, pkk = 0;
    unsigned long long pol = 0;
    if (warp == kProdWarp && lane == 0) {
        pol = l2_evict_first();
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap)) : "memory");
        for (; issued < kS && issued < nstage; ++issued) {
            issue_stage(p, G, ring, bar, prb, pkk, issued, pol);
            if (++pkk == kwu) { pkk = 0; ++prb; }
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
        // ------------------------------------------------ dequantisation: stages j, j + 4, ...
        const int q = warp & 3, j = warp >> 2;
        const int trb = 2 * q + (lane >> 4), rit = lane & 15;   // this thread's row: tile of the block, row
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const __half2 off_lo = as_h2(0x64086408u), off_hi = as_h2(0x64806480u);   // 1032, 1152
        // group j takes the pairs j, j + 4, ...; pair g is units 2 pp, 2 pp + 1 (those < kwu) of row
        // block rb = g / npr, and uses A slot g % kA
        uint32_t nfree = 0;   // waits on this group's AFreeG so far
        for (int g = j; g < npair; g += kGroups) {
            const int rb = g / npr, pp = g - rb * npr, a = g % kA;
            const int nu = ps;
            // the slot's previous group of units (g - kA) has been multiplied; the fence orders this
            // warp's tensor-memory stores below after the MMAs' reads that the wait has seen end
            if (g >= kA && !warp_wait(bar + (kAFreeG + j) * 8, nfree++ & 1u, p, abt, 2000 + g)) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const bool warp_rows = rb * kRB + 2 * q < T;       // the warp's first tile exists
            const bool mine = rb * kRB + trb < T;              // this thread's tile exists
            bool ok = true;
            for (int u = 0; u < nu; ++u) {
                const int st = rb * kwu + ps * pp + u, slot = st % kS;
                if (!warp_wait(bar + (kSFull + slot) * 8, (uint32_t)(st / kS) & 1u, p, abt, 1000 + st)) {
                    ok = false;
                    break;
                }
                uint4 cw[4] = {};
                uint2 sc = make_uint2(0u, 0u);
                if (mine) {
                    const unsigned char* unit = ring + (size_t)slot * kStageBytes + (size_t)trb * kUnitBytes;
#pragma unroll
                    for (int qb = 0; qb < 4; ++qb) cw[qb] = *reinterpret_cast<const uint4*>(unit + (qb * 16 + rit) * 16);
                    sc = *reinterpret_cast<const uint2*>(unit + 1024 + rit * 8);
                }
                __syncwarp();
                if (lane == 0) arrive(bar + (kSFree + slot) * 8);   // the stage's codes are in registers
                if (warp_rows) {
                    const uint32_t ta = tb + lane_base + kACol + (uint32_t)(64 * kPair) * (uint32_t)a + 64u * (uint32_t)u;
#pragma unroll
                    for (int half = 0; half < 2; ++half) {   // blocks 2 half, 2 half + 1: 32 columns
                        uint32_t v[32];
                        const uint32_t sw = half ? sc.y : sc.x;
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const uint4 c4 = cw[2 * half + e];
                            const __half2 d2 = e ? __high2half2(as_h2(sw)) : __low2half2(as_h2(sw));
                            const uint32_t ws[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                const uint32_t w = ws[t], w8 = w >> 8;
                                v[(e * 4 + t) * 4 + 0] = as_u32(__hmul2(__hsub2(as_h2((w & 0x000F000Fu) | 0x64006400u), off_lo), d2));
                                v[(e * 4 + t) * 4 + 1] = as_u32(__hmul2(__hsub2(as_h2((w8 & 0x000F000Fu) | 0x64006400u), off_lo), d2));
                                v[(e * 4 + t) * 4 + 2] = as_u32(__hmul2(__hsub2(as_h2((w & 0x00F000F0u) | 0x64006400u), off_hi), d2));
                                v[(e * 4 + t) * 4 + 3] = as_u32(__hmul2(__hsub2(as_h2((w8 & 0x00F000F0u) | 0x64006400u), off_hi), d2));
                            }
                        }
                        asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
                                     "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
                                     ::"r"(ta + 32u * (uint32_t)half), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]),
                                       "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]),
                                       "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
                                       "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]),
                                       "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31]) : "memory");
                    }
                }
            }
            if (!ok) break;
            if (warp_rows) asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) arrive(bar + (kAFull + a) * 8);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------ MMA issue (one lane)
        if (lane == 0) {
            // B descriptors: K-major core matrices, 512 bytes between the K halves of a step, 128
            // between 8-column groups; step ks of unit kk starts (16 kk + 2 ks) x 512 bytes in
            const uint32_t bbase = su32(bsm);
            const unsigned long long desc0 = (unsigned long long)((bbase & 0x3FFFFu) >> 4) |
                                             ((unsigned long long)(512u >> 4) << 16) |
                                             ((unsigned long long)(128u >> 4) << 32) | (1ull << 46);
            int rb = 0, pp = 0, a = 0;
            uint32_t aph = 0;   // phase parity of the A slots' current round
            for (int g = 0; g < npair; ++g) {
                const int d = rb & 1, kk0 = ps * pp;
                const int nu = ps;
                if (pp == 0 && rb >= 2 &&
                    !tc_wait(bar + (kDFree + d) * 8, (uint32_t)((rb >> 1) - 1) & 1u, p, abt, 3000 + rb))
                    break;
                if (!tc_wait(bar + (kAFull + a) * 8, aph, p, abt, 4000 + g)) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t dbase = tb + kDCols * (uint32_t)d, abase = tb + kACol + (uint32_t)(64 * kPair) * (uint32_t)a;
                for (int u = 0; u < nu; ++u) {
                    const unsigned long long dk = desc0 + (unsigned long long)((kk0 + u) * 16 * 32);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t acc = (kk0 + u > 0 || ks >= kAcc) ? 1u : 0u;   // each accumulator's first MMA overwrites
                        asm volatile("{\n .reg .pred pa;\n setp.ne.u32 pa, %4, 0;\n"
                                     " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, pa;\n}"
                                     ::"r"(dbase + 32u * (uint32_t)(ks % kAcc)), "r"(abase + 64u * (uint32_t)u + 8u * (uint32_t)ks),
                                       "l"(dk + (unsigned long long)(ks * 2 * 32)), "r"(kIdesc), "r"(acc) : "memory");
                    }
                }
                if (g + kA < npair)   // the group that takes this slot next may write it
                    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                                 ::"r"(bar + (kAFreeG + (g + kA) % kGroups) * 8) : "memory");
                if (kk0 + nu == kwu)
                    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                                 ::"r"(bar + (kDFull + d) * 8) : "memory");
                if (++pp == npr) { pp = 0; ++rb; }
                if (++a == kA) { a = 0; aph ^= 1u; }
            }
            // every MMA issued has completed before the tensor memory is released
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                         ::"r"(bar + kDone * 8) : "memory");
            tc_wait(bar + kDone * 8, 0u, p, nullptr, 7000);
        }
        __syncwarp();
    } else if (warp == kProdWarp) {
        // ------------------------------------------------ bulk copies (one lane)
        if (lane == 0) {
            for (; issued < nstage; ++issued) {
                const int slot = issued % kS;
                if (!tc_wait(bar + (kSFree + slot) * 8, (uint32_t)(issued / kS - 1) & 1u, p, abt, 5000 + issued)) break;
                issue_stage(p, G, ring, bar, prb, pkk, slot, pol);
                if (++pkk == kwu) { pkk = 0; ++prb; }
            }
            issued_stages = issued;
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue: drain, partials, ticket merge
        const int q = warp & 3, e = q * 32 + lane;
        const int trb = 2 * q + (lane >> 4), rit = lane & 15;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        for (int rb = 0; rb < nrb; ++rb) {
            const int d = rb & 1;
            // a failed wait sets the abort flag before the barrier below: every epilogue warp then
            // sees it through epi_stop and leaves together (the named barriers need all four)
            if (warp_wait(bar + (kDFull + d) * 8, (uint32_t)(rb >> 1) & 1u, p, abt, 6000 + rb)) {
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const int tl = rb * kRB + trb;
                const size_t R = (size_t)p.M.ntile * 16;   // partial rows per window and column
                float* dst = p.part + (size_t)G.w * kMaxCols * R + (size_t)(G.T0 + tl) * 16 + rit;
#pragma unroll
                for (int h = 0; h < 2; ++h) {   // 16 batch columns at a time
                    float f[16];
#pragma unroll
                    for (int ac = 0; ac < kAcc; ++ac) {   // the set's accumulators, summed in order
                        uint32_t v[16];
                        tmem_ld16(tb + lane_base + kDCols * (uint32_t)d + 32u * (uint32_t)ac + 16u * (uint32_t)h, v);
#pragma unroll
                        for (int i = 0; i < 16; ++i) f[i] = ac == 0 ? __uint_as_float(v[i]) : f[i] + __uint_as_float(v[i]);
                    }
                    if (tl < T) {   // per column, a half warp stores 16 consecutive rows
#pragma unroll
                        for (int c = 0; c < 16; ++c) dst[(size_t)(16 * h + c) * R] = f[c];
                    }
                }
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                __syncwarp();
                if (lane == 0) arrive(bar + (kDFree + d) * 8);
                __threadfence();   // this thread's partial stores visible at gpu scope before the ticket
            }
            epi_sync();   // every epilogue thread's fenced partial stores before thread 0's ticket below
            if (e == 0) {
                const int stop = *reinterpret_cast<volatile int*>(abt);
                epi_stop = stop;
                int last = 1;   // one window: this CTA has the whole sum
                if (!p.kernel_merge && G.nwin > 1) last = 0;   // merge_kernel adds the windows
                else if (!stop && G.nwin > 1) {
                    int t;
                    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                                 : "=r"(t) : "l"(p.tickets + (size_t)G.rg * p.maxrb + rb) : "memory");
                    last = t == G.nwin - 1;
                }
                merge_flag = last;
            }
            epi_sync();
            if (epi_stop) break;
            if (merge_flag) {
                if (p.epi == QL_EPI_SILU_MUL) merge_rb<true>(p, G, rb, e);
                else merge_rb<false>(p, G, rb, e);
                if (e == 0 && G.nwin > 1) p.tickets[(size_t)G.rg * p.maxrb + rb] = 0;   // re-armed for the next call
            }
            epi_sync();   // merge_flag and epi_stop are read by every epilogue thread before they change
        }
    }
    persist::stamp(tr, 3);
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    persist::stamp(tr, 4);
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tb), "r"(kTmemCols) : "memory");
    }
    // copies still in flight (only after an abort): the last use of each slot lands before the
    // CTA leaves (bounded)
    if (warp == kProdWarp && lane == 0) {
        const int n = issued_stages;
        for (int s = n - kS < 0 ? 0 : n - kS; s < n; ++s)
            tc_wait(bar + (kSFull + s % kS) * 8, (uint32_t)(s / kS) & 1u, p, nullptr, 8000 + s);
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

// Workspace: a fixed region of row-block tickets (tcgen05 form; zero between calls, whatever
// the shape, so that calls of different shapes can take turns on one workspace), then the
// windows' partial sums.
constexpr size_t kTicketInts = 65536;
struct BatchedLayout {
    int nwin, ngr, maxrb;
    size_t part_off, total;
};
static BatchedLayout batched_layout(int ntile, int nblk) {
    BatchedLayout L = {};
    batched_split(nblk, ntile, num_sms(), L.nwin, L.ngr);
    const int max_tiles = (ntile + L.ngr - 1) / L.ngr;
    L.maxrb = (max_tiles + batched::tc::kRB - 1) / batched::tc::kRB;
    L.part_off = kTicketInts * sizeof(int);
    L.total = L.part_off + (size_t)L.nwin * ntile * 16 * batched::kMaxCols * sizeof(float);
    if ((size_t)L.ngr * L.maxrb > kTicketInts) L.total = 0;   // more row blocks than tickets
    return L;
}

size_t batched_gemv_workspace_bytes(int rows, int nblk, int silu) {
    const int ntile = silu ? (rows / 2 + 7) / 8 : (rows + 15) / 16;
    return batched_layout(ntile, nblk).total;
}

// cuTensorMapEncodeTiled from the driver (no link-time dependency on libcuda).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
static EncodeTiledFn encode_tiled() {
    static const EncodeTiledFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// The stream of M as a 3-D tensor for the tcgen05 form's stage copies: [tile][unit][144 x 8 bytes]
// (a unit is 1152 bytes), boxes of one unit of 8 consecutive tiles.
static int stream_tensor_map(const PMat& M, CUtensorMap* map) {
    const EncodeTiledFn enc = encode_tiled();
    if (enc == nullptr) return set_error(QL_ECUDA, "batched gemv: cuTensorMapEncodeTiled is not available");
    const int nst = M.nblk / batched::kUnitBlocks;
    const cuuint64_t dims[3] = {(cuuint64_t)(batched::kUnitBytes / 8), (cuuint64_t)nst, (cuuint64_t)M.ntile};
    const cuuint64_t strides[2] = {(cuuint64_t)batched::kUnitBytes, (cuuint64_t)nst * batched::kUnitBytes};
    const cuuint32_t box[3] = {(cuuint32_t)(batched::kUnitBytes / 8), 1u, (cuuint32_t)batched::tc::kRB};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<uint8_t*>(M.stream), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? QL_OK : set_error(QL_ECUDA, "batched gemv: tensor map encoding failed (" + std::to_string((int)r) + ")");
}

int q4_stream_tensor_map(const PMat& M, CUtensorMap* map) { return stream_tensor_map(M, map); }

int rms_norm_launch(const float* x, int cols, float eps, const float* w, __half* xn, int T, cudaStream_t s, bool pdl) {
    const cudaError_t e = ql::launch(batched::rms_norm_kernel, dim3(T), dim3(batched::kNormT), 0, s, pdl, x, cols, eps, w, xn);
    return e == cudaSuccess ? QL_OK : cuda_error(e, "rms norm launch");
}

int f16_rows_tensor_map(const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer,
                        CUtensorMap* map, bool swizzle128) {
    const EncodeTiledFn enc = encode_tiled();
    if (enc == nullptr) return set_error(QL_ECUDA, "tensor map: cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    const cuuint64_t strides[1] = {(cuuint64_t)(inner * 2)};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? QL_OK : set_error(QL_ECUDA, "tensor map: f16 rows encoding failed (" + std::to_string((int)r) + ")");
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
    return batched_gemv_launch_traced(a, nullptr, s, pdl);
}

int batched_gemv_launch_traced(const StreamGemvArgs& a, unsigned long long* merge_trace, cudaStream_t s, bool pdl) {
    QL_REQUIRE(a.M.stream && batched_gemv_shape_ok(a.M.nblk),
               "batched gemv: cols must be 128, 256, ..., 896 or a multiple of 1024");
    QL_REQUIRE(a.batch >= 1 && a.batch <= batched::kMaxCols, "batched gemv: batch must be in [1, 32]");
    QL_REQUIRE(a.rms ? (a.xf && a.norm_w && a.xn) : a.x16 != nullptr, "batched gemv: null input");
    QL_REQUIRE(a.y && a.sync && a.workspace, "batched gemv: null output or workspace");
    const size_t need = batched_gemv_workspace_bytes(a.M.rows, a.M.nblk, a.M.silu);
    QL_REQUIRE(need > 0 && a.workspace_bytes >= need, "batched gemv: workspace too small");
    QL_REQUIRE(a.epilogue != kEpiArgmax || a.keys, "batched gemv: argmax needs keys");
    QL_REQUIRE((a.epilogue == QL_EPI_SILU_MUL) == (a.M.silu != 0), "batched gemv: SiLU*up needs a matrix packed for it");
    DevError* err = device_error_record();
    if (!err) return set_error(QL_ECUDA, "batched gemv: no device error record");
    if (int rc = batched_gemv_prepare()) return rc;
    const BatchedLayout L = batched_layout(a.M.ntile, a.M.nblk);
    const int nwin = L.nwin, ngr = L.ngr;
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
    p.part = reinterpret_cast<float*>(static_cast<char*>(a.workspace) + L.part_off);
    p.ngr = ngr;
    p.tickets = static_cast<int*>(a.workspace);
    p.maxrb = L.maxrb;
    p.trace = a.trace;
    p.mtrace = merge_trace;
    // the RMSNorm folded into the merges (merge_kernel runs in the mma.sync form only); the
    // producer's rows must come in whole warps of 32 (its chunk sums are warp reductions)
    static const bool fold_off = [] {   // QL_BATCHED_NORM_FOLD=0: rms_norm_kernel (A/B measurements)
        const char* e = std::getenv("QL_BATCHED_NORM_FOLD");
        return e != nullptr && std::atoi(e) == 0;
    }();
    const bool fold = !use_tc() && !fold_off;
    const bool consume = a.rms && a.ssq_in != nullptr && fold;
    const bool produce = a.ssq_out != nullptr && a.w_next != nullptr && a.xn != nullptr &&
                         a.epilogue == QL_EPI_ADD_RESIDUAL && fold && a.M.rows % 32 == 0 && !a.M.silu;
    if (consume) {
        p.ssq_in = a.ssq_in;
        p.eps = a.eps;
    }
    if (produce) {
        p.ssq_out = a.ssq_out;
        p.w_next = a.w_next;
        p.xn_out = a.xn;
    }
    if (a.rms && !consume) {   // the RMSNorm'd activations of every column, once, for all CTAs
        const cudaError_t e0 = ql::launch(batched::rms_norm_kernel, dim3(a.batch), dim3(batched::kNormT), 0, s, pdl,
                                          a.xf, a.M.nblk * 32, a.eps, a.norm_w, a.xn);
        if (e0 != cudaSuccess) return cuda_error(e0, "rms norm launch");
    }
    const int nt = (a.batch + 7) / 8, grid = nwin * ngr;
    cudaError_t e;
    if (use_tc()) {
        // the K windows merged by merge_kernel (default: measured faster on the batch-32 step than
        // the in-kernel ticket merge, whose merging CTA becomes the launch's tail);
        // QL_TC_KERNEL_MERGE=1 merges them inside the kernel
        static const int env_km = [] {
            const char* ev = std::getenv("QL_TC_KERNEL_MERGE");
            return ev != nullptr && std::atoi(ev) != 0 ? 1 : 0;
        }();
        p.kernel_merge = env_km;
        if (int rc = stream_tensor_map(a.M, &p.tmap)) return rc;
        e = ql::launch(batched::tc::gemv_tc_kernel, dim3(grid), dim3(batched::tc::kThreads), batched::tc::kSmem, s,
                       pdl, p);
        if (e != cudaSuccess) return cuda_error(e, "batched gemv launch");
        if (env_km || nwin == 1) return QL_OK;
        e = batched::launch_merge(p, nwin, s, pdl);
        return e == cudaSuccess ? QL_OK : cuda_error(e, "batched gemv merge launch");
    }
    e = nt == 1   ? batched::run<1>(true, &p, grid, s, pdl)
        : nt == 2 ? batched::run<2>(true, &p, grid, s, pdl)
        : nt == 3 ? batched::run<3>(true, &p, grid, s, pdl)
                  : batched::run<4>(true, &p, grid, s, pdl);
    if (e != cudaSuccess) return cuda_error(e, "batched gemv launch");
    // the windows added up and the epilogue, one CTA per SM: in the step's graph a grid of two
    // per SM ran as two waves (the second wave's CTAs passed their wait only when the first
    // wave's were done), so a larger grid only lengthens the merge
    e = batched::launch_merge(p, nwin, s, pdl);
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
