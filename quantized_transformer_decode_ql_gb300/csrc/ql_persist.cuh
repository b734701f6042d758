// Persistent decode step: the whole step of a batch of 1-2 sequences as ONE cooperative kernel.
//
// [IL] inferencelayer cuda_llm.rs, CudaQwen3::step (the step's dataflow: RMSNorm -> q|k|v ->
// qk-norm + RoPE -> paged attention -> o + residual -> RMSNorm -> gate|up -> SiLU*up -> down +
// residual; final norm, lm_head and greedy argmax; q4_0 weights with one GEMV per projection
// group); [FK] ferrum-kernels cuda_decode.rs (split-K paged decode attention over 16-token
// blocks of an f16 pool, valid length = position + 1).
//
// Why (GB300). At batch 1 a step streams 4.26 GB of q4_0 weights through 5 dependent phases per
// layer. As separate launches each phase pays a ramp and a tail: a 10-60 MB stream reaches only
// 2-4.6 TB/s of the ~6.7 TB/s the part sustains. Here one CTA per SM runs the whole step:
//  * every warp owns a fixed sequence of weight "units" (16 rows x 4 q4_0 blocks: 1 KB of codes
//    plus 128 B of scales) over ALL the step's matrices and streams them through a private
//    shared-memory ring, one bulk copy (TMA) per unit completing on the slot's mbarrier; the
//    matrices are re-laid once into a tile stream layout in which every unit is contiguous.
//    (Per-lane 16-byte cp.async copies from the row-major layout, measured first, sustained
//    only ~26 GB/s per SM.) Weights do not depend on activations, so the ring fills with the
//    next phase's weights while the CTA waits at a grid barrier, stages activations or runs
//    attention: HBM keeps streaming across phase boundaries;
//  * phases are separated by a grid-wide barrier (a counter in global memory, bounded wait:
//    after a timeout the CTA records an error, raises an abort flag and leaves the step);
//  * a matrix is split over CTAs by 16-row tiles, and inside a CTA over the 16 warps by flat
//    (tile, 4-block group) units, so every warp streams the same number of bytes; a tile shared
//    by several warps is reduced in shared memory in warp order (deterministic), the others are
//    finished from registers;
//  * the GEMV arithmetic: activations staged once per CTA as 16-bit fixed point with one
//    power-of-two scale per 32-element block; the codes masked into bytes (q and 16 q) and
//    multiplied by dp2a, so that the products and each block's sum are exact integers; the -8
//    offset enters as a staged per-block term; per row and block one I2F, FMUL and FFMA apply the
//    f16 scale and the activation scale in f32 (gemv_phase);
//  * attention: one CTA per (sequence, kv head, split), each warp one 16-token block at a
//    time. K is loaded straight into MMA fragments with 16-byte loads (head_dim permuted the
//    same way in Q and K, which leaves the dot products unchanged), S = Q K^T on mma.sync,
//    online softmax in the exp2 domain, P.V on the CUDA cores with coalesced V rows; warps merge
//    in shared memory, splits merge in the CTA that finishes last (atomic ticket, no waiting).
#pragma once

#include <cuda_fp16.h>
#include <math.h>

#include "ql_internal.h"

namespace ql {
namespace persist {

constexpr int kW = 16;                  // warps per CTA
constexpr int kT = kW * 32;             // threads per CTA
constexpr int kStages = 2;              // ring slots per warp
constexpr int kSlotUnits = 4;           // units per slot (one bulk copy)
constexpr int kUnitBlocks = 4;          // q4_0 blocks per row in one unit
constexpr int kUnitBytes = kUnitBlocks * 16 * 16 + 16 * kUnitBlocks * 2;   // 1152
constexpr int kSlotBytes = kSlotUnits * kUnitBytes;
constexpr int kRingBytes = kW * kStages * kSlotBytes;
constexpr int kBS = 16;                 // tokens per KV block
constexpr int kMaxB = kPersistMaxBatch;
constexpr int kMaxSplit = 256;
constexpr int kPartBytes = kW * 2 * 32 * 16;   // per-warp partial fragments of shared tiles
constexpr int kTraceWords = 8;                 // trace entries per (row, CTA)
constexpr int kFastSpins = 4096;               // polls of a wait before its clock starts
constexpr uint32_t kSuspendNs = 2000;          // suspend-time hint of one mbarrier poll

enum Epi { kEpiF32 = 0, kEpiResid = 1, kEpiSilu = 2, kEpiLogits = 3 };

// Shared memory behind the rings: the GEMV staging (activations, offset terms, partials) or
// the attention merge buffers, whichever is larger.
// GEMV staging per batch column: the 16-bit activations ((max_nblk * 4 + 4) x 16 B) and the
// per-block offset terms and scales ((max_nblk + 4) x 8 B); then the warps' parked tile partials.
__host__ __device__ constexpr size_t gemv_region_bytes(int batch, int max_nblk, int warps = kW) {
    return (size_t)batch * (max_nblk * 4 + 4) * 16 + (size_t)batch * (max_nblk + 4) * 8 + (size_t)warps * 2 * 32 * 16;
}
__host__ __device__ constexpr size_t attn_region_bytes(int head_dim, int group) {
    return (size_t)kW * (group * head_dim > 128 ? group * head_dim : 128) * 4 + (size_t)2 * kW * group * 4;
}

__device__ __forceinline__ __half2 as_h2(uint32_t u) {
    __half2 h;
    *reinterpret_cast<uint32_t*>(&h) = u;
    return h;
}
__device__ __forceinline__ uint32_t as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

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

// Two-way dot product of two signed 16-bit activations (a) with two unsigned bytes of b (bytes
// 0-1 for .lo, 2-3 for .hi), accumulated exactly in 32 bits: c + a.h0 * b.bk + a.h1 * b.bk+1.
__device__ __forceinline__ int dp2a_lo(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp2a_hi(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Four-way dot product of four signed bytes (a) with four unsigned bytes (b), accumulated
// exactly in 32 bits.
__device__ __forceinline__ int dp4a_su(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// ------------------------------------------------------------------------------ grid barrier
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Thread 0 stamps step `i` of the current phase (trace entries 2..5), when tracing.
__device__ __forceinline__ void stamp(unsigned long long* tr, int i) {
    if (tr != nullptr && threadIdx.x == 0) tr[i] = global_ns();
}
__device__ __forceinline__ unsigned int load_acquire(const unsigned int* a) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
    return v;
}

// Barrier over the co-resident CTAs of the launch. sync[0] counts arrivals over the whole
// launch (the k-th barrier waits for k * gridDim.x of them, plus p.barrier_extra, which only a
// test sets: an arrival that never comes); sync[2] is the abort flag. The wait is bounded by the
// clock: after p.barrier_timeout_ns the CTA records an error, raises the flag and returns false,
// as does every CTA that sees the flag; the caller then leaves the step. With p.trace set,
// thread 0 stamps its arrival and its exit (globaltimer, ns) in row k of the trace (entries 0
// and 1 of kTraceWords; the phase that ends at barrier k stamps its own steps in 2..5).
static __device__ __noinline__ bool grid_barrier(const PersistParams& p, unsigned int& target, int* ok_smem) {
    __syncthreads();
    if (threadIdx.x == 0) {
        target += gridDim.x;
        unsigned long long* tr =
            p.trace ? p.trace + ((size_t)(target / gridDim.x) * gridDim.x + blockIdx.x) * kTraceWords : nullptr;
        if (tr) tr[0] = global_ns();
        const unsigned int need = target + p.barrier_extra;
        int ok = 1;
        // release: the CTA's writes (ordered before this by the bar.sync above) become visible
        // to every CTA whose acquire load reads the count
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p.sync) : "memory");
        for (int spin = 0; spin < kFastSpins && load_acquire(p.sync) < need; ++spin) {
        }
        if (load_acquire(p.sync) < need) {
            const unsigned long long t0 = global_ns();
            for (unsigned int spin = 1;; ++spin) {
                if (load_acquire(p.sync) >= need) break;
                if ((spin & 15u) == 0) {
                    if (load_acquire(p.sync + 2) != 0u) {
                        ok = 0;
                        break;
                    }
                    if (global_ns() - t0 > p.barrier_timeout_ns) {
                        record_device_error(p.err, kErrStepBarrier, (long long)(target / gridDim.x),
                                            (long long)blockIdx.x);
                        atomicExch(p.sync + 2, 1u);
                        ok = 0;
                        break;
                    }
                }
            }
        }
        if (tr) tr[1] = global_ns();
        *ok_smem = ok;
    }
    __syncthreads();
    return *ok_smem != 0;
}

// Every CTA calls this once, last. The CTA that leaves last re-arms the counters for the next
// launch (all others are past their last wait by then); after an abort it also clears the
// attention tickets, which an interrupted phase may have left counted.
static __device__ void leave_step(const PersistParams& p) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(p.sync + 1, 1u) == gridDim.x - 1) {
            if (atomicAdd(p.sync + 2, 0u) != 0u)
                for (int i = 0; i < p.B * p.nkv; ++i) atomicExch(p.tickets + i, 0);
            atomicExch(p.sync, 0u);
            atomicExch(p.sync + 2, 0u);
            __threadfence();
            atomicExch(p.sync + 1, 0u);
        }
    }
}

// ------------------------------------------------------------------------------ weight ring
// The step's matrices in streaming order: 4 per layer (q|k|v, o, gate|up, down), then lm_head.
// The kernel copies their descriptors into shared memory (`mats`) once at the start.
__device__ __forceinline__ PMat mat_global(const PersistParams& p, int wp) {
    return wp < 4 * p.n_layers ? p.layers[wp >> 2].m[wp & 3] : p.lm;
}
__host__ __device__ constexpr size_t mat_table_bytes(int n_layers) { return (size_t)(4 * n_layers + 1) * sizeof(PMat); }
// Tiles [t0, t1) of a matrix handled by this CTA (balanced to one tile; ntile * grid < 2^32).
__device__ __forceinline__ void cta_tiles(int ntile, int& t0, int& t1) {
    t0 = (int)((blockIdx.x * (unsigned)ntile) / gridDim.x);
    t1 = (int)(((blockIdx.x + 1) * (unsigned)ntile) / gridDim.x);
}
// First unit of warp w among the U units of its CTA of W warps (balanced to one unit).
template <int W>
__device__ __forceinline__ int warp_unit(int U, int w) { return (w * U) / W; }

// Global row of row r (0..15) of a tile; rows past the matrix read row 0 and are discarded.
__device__ __forceinline__ int tile_row(const PMat& M, int tile, int r, bool& ok) {
    if (M.silu) {
        const int half = M.rows >> 1, i = tile * 8 + (r & 7);
        ok = i < half;
        return ok ? (r < 8 ? i : half + i) : 0;
    }
    const int row = tile * 16 + r;
    ok = row < M.rows;
    return ok ? row : 0;
}

// Issue side of a warp's ring. The matrices are stored in the tile stream layout
// (stream_pack_kernel): unit (tile, k) is 1152 contiguous bytes at stream + (tile nst + k) 1152,
// codes [block 0..3][row 0..15] x 16 B, then the 16 rows' 4 scales (8 B each), so a warp's
// units of one matrix are one contiguous byte range. Lane 0 copies up to kSlotUnits units at a
// time into a ring slot with one bulk copy (TMA, cp.async.bulk) that completes on the slot's
// mbarrier (a copy never crosses the end of the warp's range in a matrix). A bulk copy costs its
// issuing warp a fixed time, so copies of several units stream faster than one unit each.
struct Ring {
    int wp, nmat;          // matrix of the next copy; nmat = end of the step
    int u, u_end;          // unit (within the warp's range of that matrix) and range end
    int ubase;             // the CTA's first unit in the matrix (routed experts)
    const uint8_t* src;    // stream address of unit u (not used for routed experts)
    unsigned int issued, consumed;   // slots; ring slot = count % kStages
    uint32_t base;         // shared-memory address of this warp's ring
    uint32_t mbar;         // shared-memory address of this warp's kStages mbarriers
    int dead;              // a wait ran out: issue and wait no more (the step is aborted)
};

// Move to the first matrix at or after r.wp in which this warp (of W) has units.
template <int W>
__device__ __forceinline__ void ring_seek(Ring& r, const PMat* mats, int warp) {
    for (; r.wp < r.nmat; ++r.wp) {
        const PMat& M = mats[r.wp];
        int t0, t1;
        cta_tiles(M.ntile, t0, t1);
        const int nst = M.nblk / kUnitBlocks;
        const int U = (t1 - t0) * nst;
        const int u0 = warp_unit<W>(U, warp), u1 = warp_unit<W>(U, warp + 1);
        if (u1 > u0) {
            r.u = u0;
            r.u_end = u1;
            r.ubase = t0 * nst;
            // routed experts: the address depends on the selection, read when the copy is issued
            r.src = M.sel ? nullptr : M.stream + ((size_t)t0 * nst + u0) * kUnitBytes;
            return;
        }
    }
}

// Copy the next slot's units (up to kSlotUnits, not past the warp's range end).
template <int W, bool SEL = false>
__device__ __forceinline__ void ring_issue(Ring& r, const PMat* mats, int warp, int lane) {
    if (r.wp >= r.nmat || r.dead) return;
    int n = min(kSlotUnits, r.u_end - r.u);
    if (SEL) {
        const PMat& M = mats[r.wp];
        // the selected expert's run of units; a copy stops at the expert's end. An id outside
        // the experts (not one a router writes) reads expert 0 instead of leaving the stream.
        const int per = M.etiles * (M.nblk / kUnitBlocks);
        const int abs = r.ubase + r.u, j = abs / per, within = abs - j * per;
        int e = M.sel[j];
        if (e < 0 || e >= M.nexp) e = 0;
        n = min(n, per - within);
        r.src = M.stream + ((size_t)e * per + within) * kUnitBytes;
    }
    if (lane == 0) {
        const unsigned int slot = r.issued % kStages;
        const uint32_t mb = r.mbar + slot * 8, dst = r.base + slot * kSlotBytes;
        const uint32_t bytes = (uint32_t)(n * kUnitBytes);
        // order this warp's earlier generic-proxy reads of the slot before the async-proxy write
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mb), "r"(bytes) : "memory");
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
                     ::"r"(dst), "l"(r.src), "r"(bytes), "r"(mb), "l"(l2_evict_first()) : "memory");
    }
    r.src += (size_t)n * kUnitBytes;
    ++r.issued;
    r.u += n;
    if (r.u == r.u_end) {
        ++r.wp;
        ring_seek<W>(r, mats, warp);
    }
}

// Test (and wait a while for) the completion of phase `parity` of an mbarrier: the hardware
// suspends the warp until the phase completes or about kSuspendNs pass, so waiting warps do
// not spin on issue slots that the warps with data need.
__device__ __forceinline__ bool mbar_test(uint32_t mb, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred q;\n mbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2, %3;\n selp.u32 %0, 1, 0, q;\n}"
        : "=r"(done)
        : "r"(mb), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return done != 0;
}

// Wait until unit n (n >= r.consumed) has landed in its slot. Bounded by the clock: when the
// bound runs out the warp records an error, raises the step's abort flag and stops using the
// ring.
__device__ __forceinline__ void ring_wait(Ring& r, const PersistParams& p, unsigned int n) {
    if (r.dead) return;
    const uint32_t mb = r.mbar + (n % kStages) * 8, parity = (n / kStages) & 1u;
    // fast path without the clock (reading %globaltimer is slow); the clock bounds the rest
    for (int spin = 0; spin < kFastSpins; ++spin)
        if (mbar_test(mb, parity)) return;
    const unsigned long long t0 = global_ns();
    for (unsigned int spin = 1;; ++spin) {
        if (mbar_test(mb, parity)) return;
        if ((spin & 63u) == 0 && global_ns() - t0 > p.barrier_timeout_ns) break;
    }
    if ((threadIdx.x & 31) == 0) {
        record_device_error(p.err, kErrGemvStage, blockIdx.x, (long long)n);
        atomicExch(p.sync + 2, 1u);
    }
    r.dead = 1;
}

// ------------------------------------------------------------------------------ GEMV phase
// Scalars of the step that a GEMV phase reads after its wait on the predecessor, passed by value:
// read through the reference to the kernel parameters they were a cold load on the critical
// path of every launch (the kernel reads them before its wait, see hot_scalars).
struct Hot {
    int B, max_nblk;
    float eps;
};
__device__ __forceinline__ Hot hot_scalars(const PersistParams& p) {
    Hot h{p.B, p.max_nblk, p.eps};
    // opaque to the compiler from here on: kept in registers, not re-read after the wait
    asm volatile("" : "+r"(h.B), "+r"(h.max_nblk), "+f"(h.eps));
    return h;
}
// Stage the activations of all B columns as 16-bit fixed point, one power-of-two scale per
// 32-element block: x_int = rint(x 2^s), with s the largest shift that keeps the block's largest
// |x| (times 1.001, a margin for the rounding) below 2^15. The scaling is exact; the rounding is
// the only error, at most 2^-(s+1) per element, relative 2^-15 of the block's largest value. Per
// column and block j: 4 chunks of 16 bytes (chunk t: int16 pairs (x[4t], x[4t+1]), (x[4t+2],
// x[4t+3]), (x[16+4t], x[17+4t]), (x[18+4t], x[19+4t]) of the block's elements: the order in which
// code word t holds their nibbles), and the block's pair (-128 sum_e x_int[e], 2^-(s+4)): the
// offset term of the codes' -8 (times the 16 of the high nibbles' scale, see gemv_phase) and the
// factor that undoes both scalings. rint is the round-to-nearest-even of an FFMA that adds
// 1.5 * 2^23, whose low 16 bits are then the integer. RMS: the input is the f32 residual stream,
// normalised (RMSNorm with weight w) on the way; the first kHeld items of a thread and their
// weights stay in registers between the two passes. f16 input: kHeld items per thread are loaded
// together. The 4 chunks of a block are 4 consecutive items (lanes 4k..4k+3 of a warp): their
// largest magnitude and their sum take two shuffles each. Data written earlier in the launch by
// other CTAs is read with ld.global.cg (L2).
template <bool RMS, int W>
__device__ __noinline__ void stage_x(int B, float eps, int nblk, int cstride, const float* xf, const __half* x16,
                                     const float* w, uint4* xs, int2* sxs, int sxstride) {
    constexpr int kHeld = RMS ? 2 : 4, kT = W * 32;
    constexpr uint32_t kMagic = 0x4B400000u;   // bits of 1.5 * 2^23
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cols = nblk * 32, nitems = B * nblk * 4;
    const int rounds = (nitems + kT - 1) / kT;

    // item -> (column b, block j, chunk t) and its element offset
    auto where = [&](int item, int& b, int& j, int& t) -> size_t {
        t = item & 3;
        const int bj = item >> 2;
        b = bj < nblk ? 0 : (bj < 2 * nblk ? 1 : bj / nblk);   // batches of 1-2: no division
        j = bj - b * nblk;
        return (size_t)b * cols + 32 * j + 4 * t;
    };
    // the item's 8 values: elements 4t..4t+3 and 16+4t..19+4t of its block
    auto load = [&](int item, float (&v)[8]) {
        int b, j, t;
        const size_t off = where(item, b, j, t);
        if (RMS) {
            const float4 a = __ldcg(reinterpret_cast<const float4*>(xf + off));
            const float4 h = __ldcg(reinterpret_cast<const float4*>(xf + off + 16));
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            v[4] = h.x; v[5] = h.y; v[6] = h.z; v[7] = h.w;
        } else {
            const uint2 a = __ldcg(reinterpret_cast<const uint2*>(x16 + off));
            const uint2 h = __ldcg(reinterpret_cast<const uint2*>(x16 + off + 16));
            const float2 f0 = __half22float2(as_h2(a.x)), f1 = __half22float2(as_h2(a.y));
            const float2 f2 = __half22float2(as_h2(h.x)), f3 = __half22float2(as_h2(h.y));
            v[0] = f0.x; v[1] = f0.y; v[2] = f1.x; v[3] = f1.y;
            v[4] = f2.x; v[5] = f2.y; v[6] = f3.x; v[7] = f3.y;
        }
    };
    auto load_w = [&](int item, float (&v)[8]) {
        const int j = (item >> 2) % nblk, t = item & 3;
        const float4 a = __ldg(reinterpret_cast<const float4*>(w + 32 * j + 4 * t));
        const float4 h = __ldg(reinterpret_cast<const float4*>(w + 32 * j + 16 + 4 * t));
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = h.x; v[5] = h.y; v[6] = h.z; v[7] = h.w;
    };
    // fixed point of one item (all lanes of the warp call it: its shuffles pair the 4 lanes of a
    // block, which are in range together)
    auto emit = [&](int item, bool ok, const float (&v)[8]) {
        float m = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        // s = 14 - floor(log2(1.001 m)): |x| 2^s < 2^15 / 1.001 (the exponent field; a zero or
        // subnormal block gives a large s, clamped so that 2^s and 2^-(s+4) stay normal floats)
        const int e = (int)((__float_as_uint(m * 1.001f) >> 23) & 0xFFu) - 127;
        int sh = 14 - e;
        sh = sh > 100 ? 100 : (sh < -100 ? -100 : sh);
        const float sc = __uint_as_float((uint32_t)(sh + 127) << 23);
        uint32_t u[8], sum = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            u[i] = __float_as_uint(fmaf(v[i], sc, 12582912.0f));   // kMagic + rint(x 2^s)
            sum += u[i];
        }
        int n = (int)(sum - 8u * kMagic);   // the 8 integers' sum (exact: wraps back into range)
        n += __shfl_xor_sync(0xffffffffu, n, 1);
        n += __shfl_xor_sync(0xffffffffu, n, 2);
        if (ok) {
            int b, j, t;
            where(item, b, j, t);
            xs[(size_t)b * cstride + 4 * j + t] =
                make_uint4(__byte_perm(u[0], u[1], 0x5410), __byte_perm(u[2], u[3], 0x5410),
                           __byte_perm(u[4], u[5], 0x5410), __byte_perm(u[6], u[7], 0x5410));
            if (t == 0) sxs[b * sxstride + j] = make_int2(-128 * n, (int)((uint32_t)(127 - sh - 4) << 23));
        }
    };

    float hx[kHeld][8], hw[kHeld][8];
#pragma unroll
    for (int r = 0; r < kHeld; ++r)
#pragma unroll
        for (int i = 0; i < 8; ++i) hx[r][i] = hw[r][i] = 0.f;
#pragma unroll
    for (int r = 0; r < kHeld; ++r) {
        const int item = tid + r * kT;
        if (item < nitems) {
            load(item, hx[r]);
            if (RMS) load_w(item, hw[r]);
        }
    }
    float rs0 = 1.0f, rs1 = 1.0f;
    if (RMS) {
        // per column, the mean square: thread sums, warp sums, then the warps' in warp order (a
        // shared array of this function: direct shared-memory accesses); column 1 only at batch 2
        float ss0 = 0.f, ss1 = 0.f;
        const float inv_cols = 1.0f / (float)cols;   // while the loads are in flight
#pragma unroll
        for (int r = 0; r < kHeld; ++r) {
            float s2 = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) s2 = fmaf(hx[r][i], hx[r][i], s2);
            if (tid + r * kT < nblk * 4) ss0 += s2; else ss1 += s2;
        }
        for (int item = tid + kHeld * kT; item < nitems; item += kT) {
            float v[8];
            load(item, v);
            float s2 = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) s2 = fmaf(v[i], v[i], s2);
            if (item < nblk * 4) ss0 += s2; else ss1 += s2;
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) ss0 += __shfl_xor_sync(0xffffffffu, ss0, o);
        if (B > 1) {
#pragma unroll
            for (int o = 16; o; o >>= 1) ss1 += __shfl_xor_sync(0xffffffffu, ss1, o);
        }
        __shared__ float2 wsum[W];
        if (lane == 0) wsum[warp] = make_float2(ss0, ss1);
        __syncthreads();
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int i = 0; i < W; ++i) {
            const float2 v = wsum[i];
            a0 += v.x;
            a1 += v.y;
        }
        rs0 = rsqrtf(fmaf(a0, inv_cols, eps));
        rs1 = rsqrtf(fmaf(a1, inv_cols, eps));
    }
#pragma unroll
    for (int r = 0; r < kHeld; ++r) {
        if (r < rounds) {   // uniform over the CTA: every lane of a warp takes the shuffles
            const int item = tid + r * kT;
            const float rr = item < nblk * 4 ? rs0 : rs1;
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = RMS ? hx[r][i] * rr * hw[r][i] : hx[r][i];
            emit(item, item < nitems, v);
        }
    }
    for (int r = kHeld; r < rounds; ++r) {
        const int item = tid + r * kT;
        const bool ok = item < nitems;
        const float rr = item < nblk * 4 ? rs0 : rs1;
        float v[8], wv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = wv[i] = 0.f;
        if (ok) {
            load(item, v);
            if (RMS) load_w(item, wv);
        }
        if (RMS) {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] *= rr * wv[i];
        }
        emit(item, ok, v);
    }
}

// The int8 activation form ([IL] CudaQwen3::absmax: the GEMV reads its activation vector with
// one scale, xs = [max|x|, 1/max|x|]): per column, m = max|x| over the whole vector (a CTA-wide
// reduction; RMS: of |x w| times the RMSNorm scale, found with the mean square), codes
// q = rint(x * (127 / m)) with the division and the product each one f32 operation (__fdiv_rn,
// __fmul_rn, then the exact rounding of an FADD of 1.5 * 2^23). Per column and block j two
// uint4: (x[0..3], x[16..19], x[4..7], x[20..23]) and (x[8..11], x[24..27], x[12..15], x[28..31])
// as signed bytes (code word t's low and high nibbles' elements), and the block's pair
// (-128 sum_e q[e], m / (127 * 16)).
template <bool RMS, int W>
__device__ __noinline__ void stage_x8(int B, float eps, int nblk, int cstride, const float* xf, const __half* x16,
                                      const float* w, uint4* xs, int2* sxs, int sxstride) {
    constexpr int kHeld = 3, kT = W * 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cols = nblk * 32, nitems = B * nblk * 4;
    const int rounds = (nitems + kT - 1) / kT;
    auto where = [&](int item, int& b, int& j, int& t) -> size_t {
        t = item & 3;
        const int bj = item >> 2;
        b = bj < nblk ? 0 : (bj < 2 * nblk ? 1 : bj / nblk);
        j = bj - b * nblk;
        return (size_t)b * cols + 32 * j + 4 * t;
    };
    auto load = [&](int item, float (&v)[8]) {
        int b, j, t;
        const size_t off = where(item, b, j, t);
        if (RMS) {
            const float4 a = __ldcg(reinterpret_cast<const float4*>(xf + off));
            const float4 h = __ldcg(reinterpret_cast<const float4*>(xf + off + 16));
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            v[4] = h.x; v[5] = h.y; v[6] = h.z; v[7] = h.w;
        } else {
            const uint2 a = __ldcg(reinterpret_cast<const uint2*>(x16 + off));
            const uint2 h = __ldcg(reinterpret_cast<const uint2*>(x16 + off + 16));
            const float2 f0 = __half22float2(as_h2(a.x)), f1 = __half22float2(as_h2(a.y));
            const float2 f2 = __half22float2(as_h2(h.x)), f3 = __half22float2(as_h2(h.y));
            v[0] = f0.x; v[1] = f0.y; v[2] = f1.x; v[3] = f1.y;
            v[4] = f2.x; v[5] = f2.y; v[6] = f3.x; v[7] = f3.y;
        }
    };
    auto load_w = [&](int item, float (&v)[8]) {
        const int j = (item >> 2) % nblk, t = item & 3;
        const float4 a = __ldg(reinterpret_cast<const float4*>(w + 32 * j + 4 * t));
        const float4 h = __ldg(reinterpret_cast<const float4*>(w + 32 * j + 16 + 4 * t));
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = h.x; v[5] = h.y; v[6] = h.z; v[7] = h.w;
    };
    float hx[kHeld][8], hw[kHeld][8];
#pragma unroll
    for (int r = 0; r < kHeld; ++r)
#pragma unroll
        for (int i = 0; i < 8; ++i) hx[r][i] = hw[r][i] = 0.f;
#pragma unroll
    for (int r = 0; r < kHeld; ++r) {
        const int item = tid + r * kT;
        if (item < nitems) {
            load(item, hx[r]);
            if (RMS) load_w(item, hw[r]);
        }
    }
    // pass 1: per column the mean square (RMS) and the largest magnitude
    float ss0 = 0.f, ss1 = 0.f, mx0 = 0.f, mx1 = 0.f;
    auto account = [&](int item, const float (&v)[8], const float (&wv)[8]) {
        float s2 = 0.f, m = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (RMS) s2 = fmaf(v[i], v[i], s2);
            m = fmaxf(m, fabsf(RMS ? v[i] * wv[i] : v[i]));
        }
        if (item < nblk * 4) {
            ss0 += s2;
            mx0 = fmaxf(mx0, m);
        } else {
            ss1 += s2;
            mx1 = fmaxf(mx1, m);
        }
    };
#pragma unroll
    for (int r = 0; r < kHeld; ++r)
        if (tid + r * kT < nitems) account(tid + r * kT, hx[r], hw[r]);
    for (int item = tid + kHeld * kT; item < nitems; item += kT) {
        float v[8], wv[8];
        load(item, v);
        if (RMS) load_w(item, wv);
        account(item, v, wv);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        ss0 += __shfl_xor_sync(0xffffffffu, ss0, o);
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        ss1 += __shfl_xor_sync(0xffffffffu, ss1, o);
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    __shared__ float4 wred[W];
    if (lane == 0) wred[warp] = make_float4(ss0, ss1, mx0, mx1);
    __syncthreads();
    float a0 = 0.f, a1 = 0.f, m0 = 0.f, m1 = 0.f;
#pragma unroll
    for (int i = 0; i < W; ++i) {
        const float4 v = wred[i];
        a0 += v.x;
        a1 += v.y;
        m0 = fmaxf(m0, v.z);
        m1 = fmaxf(m1, v.w);
    }
    const float rs0 = RMS ? rsqrtf(fmaf(a0, 1.0f / (float)cols, eps)) : 1.0f;
    const float rs1 = RMS ? rsqrtf(fmaf(a1, 1.0f / (float)cols, eps)) : 1.0f;
    if (RMS) {
        m0 *= rs0;
        m1 *= rs1;
    }
    const float sc0 = m0 > 0.f ? __fdiv_rn(127.0f, m0) : 0.f, sc1 = m1 > 0.f ? __fdiv_rn(127.0f, m1) : 0.f;
    const int f0 = __float_as_int(__fdiv_rn(m0, 2032.0f)), f1 = __float_as_int(__fdiv_rn(m1, 2032.0f));
    // pass 2: codes, the blocks' offset terms (4 consecutive items = the 4 lanes of a block)
    uint2* xs2 = reinterpret_cast<uint2*>(xs);
    auto emit = [&](int item, bool ok, const float (&v)[8], float sc, int fb) {
        uint32_t u[8];
        int sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float r = __fadd_rn(__fmul_rn(v[i], sc), 12582912.0f);   // 1.5 * 2^23 + rint(x sc)
            int qv = (int)(__float_as_uint(r) - 0x4B400000u);
            qv = qv > 127 ? 127 : (qv < -127 ? -127 : qv);
            u[i] = (uint32_t)qv;
            sum += qv;
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        if (ok) {
            int b, j, t;
            where(item, b, j, t);
            const uint32_t lo = __byte_perm(__byte_perm(u[0], u[1], 0x0040), __byte_perm(u[2], u[3], 0x0040), 0x5410);
            const uint32_t hi = __byte_perm(__byte_perm(u[4], u[5], 0x0040), __byte_perm(u[6], u[7], 0x0040), 0x5410);
            xs2[(size_t)b * cstride * 2 + 4 * j + t] = make_uint2(lo, hi);
            if (t == 0) sxs[b * sxstride + j] = make_int2(-128 * sum, fb);
        }
    };
#pragma unroll
    for (int r = 0; r < kHeld; ++r) {
        if (r < rounds) {
            const int item = tid + r * kT;
            const bool first = item < nblk * 4;
            const float rr = first ? rs0 : rs1;
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = RMS ? hx[r][i] * rr * hw[r][i] : hx[r][i];
            emit(item, item < nitems, v, first ? sc0 : sc1, first ? f0 : f1);
        }
    }
    for (int r = kHeld; r < rounds; ++r) {
        const int item = tid + r * kT;
        const bool ok = item < nitems;
        const bool first = item < nblk * 4;
        const float rr = first ? rs0 : rs1;
        float v[8], wv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = wv[i] = 0.f;
        if (ok) {
            load(item, v);
            if (RMS) load_w(item, wv);
        }
        if (RMS) {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] *= rr * wv[i];
        }
        emit(item, ok, v, first ? sc0 : sc1, first ? f0 : f1);
    }
}

// Epilogue of one finished 16-row tile. acc[b][0] / acc[b][1] are this lane's sums of rows
// (lane & 7) and (lane & 7) + 8 of the tile over the blocks of its quarter (lane >> 3) of every
// unit, for column b; the quarters are added here (lanes l, l ^ 8, l ^ 16, l ^ 24), then
// lanes 0..15 hold rows 0..15 (SiLU*up:
// lane l < 8 holds gate row l and its up row l + 8). All 32 lanes of the warp call it. Out of
// line: it runs once per tile, and the unit loop stays small.
template <int NB>
__device__ __noinline__ void finish_tile(const PersistParams& p, const PMat& M, int epi, int tile,
                                         const float (&acc)[NB][2], void* y, int ld, unsigned long long (&best)[NB],
                                         int lane) {
    float v0[NB], v1[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        float a = acc[b][0], c = acc[b][1];
        a += __shfl_xor_sync(0xffffffffu, a, 8);
        c += __shfl_xor_sync(0xffffffffu, c, 8);
        a += __shfl_xor_sync(0xffffffffu, a, 16);
        c += __shfl_xor_sync(0xffffffffu, c, 16);
        v0[b] = a;
        v1[b] = c;
    }
    const int hr = lane & 15;
    if (epi == kEpiSilu) {
        const int i = tile * 8 + hr;
        if (lane < 8 && i < (M.rows >> 1)) {
            __half* act = static_cast<__half*>(y);
#pragma unroll
            for (int b = 0; b < NB; ++b) act[(size_t)b * ld + i] = __float2half_rn(silu(v0[b]) * v1[b]);
        }
        return;
    }
    const int row = tile * 16 + hr;
    if (lane < 16 && row < M.rows) {
        float* yf = static_cast<float*>(y);
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const float v = hr < 8 ? v0[b] : v1[b];
            float* dst = yf + (size_t)b * ld + row;
            if (epi == kEpiResid) {
                *dst = __ldcg(dst) + v;
            } else {
                *dst = v;
                if (epi == kEpiLogits) {
                    const unsigned long long key = argmax_key(v, row);
                    best[b] = key > best[b] ? key : best[b];
                }
            }
        }
    }
}

// One GEMV phase of the step: y = epilogue(W x) for this CTA's tiles of M, NB = batch columns.
// All threads of the CTA call it. The warp consumes its ring slots in the order the issue side
// produced them and refills each slot once its units are done. Per unit, lane (quarter
// bq = lane >> 3, rows r = lane & 7 and r + 8) takes block bq of both rows: code word t of a
// block holds the nibbles of elements 4t..4t+3 (low) and 16+4t..19+4t (high); masking it gives
// the low codes q as bytes and the high ones as bytes 16 q, and dp2a multiplies byte pairs with
// the staged int16 activation pairs, summing exactly in 32 bits (low and high apart, the high
// sum starting at the block's staged offset term -128 sum x_int). 16 lo + hi is then
// 16 sum_e (q_e - 8) x_int[e] exactly; per row and block one I2F, and an FMUL and an FFMA apply
// the f16 scale and the activation block's 2^-(s + 4) in f32. The two rows share every
// activation load. (An MMA form wastes 7 of the 8 columns of an m16n8k16 tile at batch 1-2 and
// measured slower; the f16 HFMA2 form of the same loop issued about twice the instructions.)
template <int NB, int W, bool I8 = false, bool SEL = false>
__device__ __noinline__ void gemv_phase(const PersistParams& p, Hot h, const PMat* mats, int wp, int epi, bool rms,
                                        Ring& ring, const float* xf,
                                        const __half* x16, const float* norm_w, void* y, int ld,
                                        unsigned char* region,
                                        unsigned long long (*kred)[kMaxB], unsigned long long* tr) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int bq = lane >> 3, rq = lane & 7;
    const PMat M = mats[wp];
    const int cstride = h.max_nblk * 4 + 4;   // uint4 units between staged columns (+64 B)
    const int sxstride = h.max_nblk + 4;      // block (offset, scale) pairs between staged columns
    // staged activation columns: the batch, or (routed experts' down rows) one per expert slot
    const int SB = (SEL && M.xsel) ? M.nsel : h.B;
    uint4* xs = reinterpret_cast<uint4*>(region);
    int2* sxs = reinterpret_cast<int2*>(xs + (size_t)SB * cstride);
    float4* part = reinterpret_cast<float4*>(sxs + (size_t)SB * sxstride);   // [W][2][32]

    if (I8) {
        if (rms)
            stage_x8<true, W>(SB, h.eps, M.nblk, cstride, xf, x16, norm_w, xs, sxs, sxstride);
        else
            stage_x8<false, W>(SB, h.eps, M.nblk, cstride, xf, x16, norm_w, xs, sxs, sxstride);
    } else {
        if (rms)
            stage_x<true, W>(SB, h.eps, M.nblk, cstride, xf, x16, norm_w, xs, sxs, sxstride);
        else
            stage_x<false, W>(SB, h.eps, M.nblk, cstride, xf, x16, norm_w, xs, sxs, sxstride);
    }
    __syncthreads();
    stamp(tr, 2);

    Ring r = ring;   // a register copy for the loop; written back at the end
    // slots not yet in flight (a kernel may issue fewer than kStages before it waits on its
    // predecessor, so that its activation loads do not queue behind a full ring)
    for (unsigned int i = r.issued - r.consumed; i < (unsigned int)kStages; ++i) ring_issue<W, SEL>(r, mats, warp, lane);
    const int nst = M.nblk / kUnitBlocks;
    int T0, T1;
    cta_tiles(M.ntile, T0, T1);
    const int U = (T1 - T0) * nst;
    const int u0 = warp_unit<W>(U, warp), u1 = warp_unit<W>(U, warp + 1);
    const unsigned char* ring_g = reinterpret_cast<const unsigned char*>(region) - (size_t)W * kStages * kSlotBytes +
                                  (size_t)warp * kStages * kSlotBytes;

    unsigned long long best[NB];
    float acc[NB][2];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        best[b] = 0ull;
        acc[b][0] = acc[b][1] = 0.f;
    }
    const int q0 = u1 > u0 ? (nst == 32 ? u0 >> 5 : u0 / nst) : 0;   // 4096-column matrices: a shift
    int tile = T0 + q0, k = u1 > u0 ? u0 - q0 * nst : 0;
    const int first_tile = tile;
    int xcol = (SEL && M.xsel) ? tile / M.etiles : 0;   // routed experts' down rows: the tile's slot

    // this lane's share of one unit (block group kk of the tile): block bq of rows rq, rq + 8
    auto unit = [&](const unsigned char* stg, int kk) {
        const uint4 c0 = *reinterpret_cast<const uint4*>(stg + (bq * 16 + rq) * 16);
        const uint4 c1 = *reinterpret_cast<const uint4*>(stg + (bq * 16 + rq + 8) * 16);
        const float d0 = __half2float(*reinterpret_cast<const __half*>(stg + kUnitBlocks * 256 + rq * 8 + 2 * bq));
        const float d1 = __half2float(*reinterpret_cast<const __half*>(stg + kUnitBlocks * 256 + (rq + 8) * 8 + 2 * bq));
        const int j = kk * kUnitBlocks + bq;
        const uint32_t w0[4] = {c0.x, c0.y, c0.z, c0.w}, w1[4] = {c1.x, c1.y, c1.z, c1.w};
        uint32_t l0[4], h0[4], l1[4], h1[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            l0[t] = w0[t] & 0x0F0F0F0Fu;
            h0[t] = w0[t] & 0xF0F0F0F0u;
            l1[t] = w1[t] & 0x0F0F0F0Fu;
            h1[t] = w1[t] & 0xF0F0F0F0u;
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const int bc = (SEL && M.xsel) ? xcol : b;   // the staged column this tile multiplies
            const int2 ov = sxs[bc * sxstride + j];
            const float f = __int_as_float(ov.y);   // the activation block's scale / 16
            int lo0 = 0, hi0 = ov.x, lo1 = 0, hi1 = ov.x;
            if (I8) {   // int8 codes: one dp4a per nibble half of a code word
                const uint4 XA = xs[(size_t)bc * cstride + 2 * j], XB = xs[(size_t)bc * cstride + 2 * j + 1];
                const uint32_t xl[4] = {XA.x, XA.z, XB.x, XB.z}, xh[4] = {XA.y, XA.w, XB.y, XB.w};
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    lo0 = dp4a_su(xl[t], l0[t], lo0);
                    lo1 = dp4a_su(xl[t], l1[t], lo1);
                    hi0 = dp4a_su(xh[t], h0[t], hi0);
                    hi1 = dp4a_su(xh[t], h1[t], hi1);
                }
            } else {
                const uint4* xb = xs + (size_t)bc * cstride + 4 * j;
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const uint4 X = xb[t];
                    lo0 = dp2a_lo(X.x, l0[t], lo0);
                    lo1 = dp2a_lo(X.x, l1[t], lo1);
                    lo0 = dp2a_hi(X.y, l0[t], lo0);
                    lo1 = dp2a_hi(X.y, l1[t], lo1);
                    hi0 = dp2a_lo(X.z, h0[t], hi0);
                    hi1 = dp2a_lo(X.z, h1[t], hi1);
                    hi0 = dp2a_hi(X.w, h0[t], hi0);
                    hi1 = dp2a_hi(X.w, h1[t], hi1);
                }
            }
            acc[b][0] = fmaf(d0 * f, (float)(lo0 * 16 + hi0), acc[b][0]);
            acc[b][1] = fmaf(d1 * f, (float)(lo1 * 16 + hi1), acc[b][1]);
        }
    };
    // after unit u: at the end of this warp's part of a tile finish the tile if the warp covered
    // all of it, else park the sums (slot 0: the warp's first tile, slot 1: its last)
    auto advance = [&](int u) {
        if (++k == nst || u + 1 == u1) {
            const int ts = (tile - T0) * nst;
            if (u0 <= ts && u + 1 == ts + nst) {
                finish_tile<NB>(p, M, epi, tile, acc, y, ld, best, lane);
            } else {
                float4 v = make_float4(acc[0][0], acc[0][1], 0.f, 0.f);
                if (NB > 1) {
                    v.z = acc[NB > 1 ? 1 : 0][0];
                    v.w = acc[NB > 1 ? 1 : 0][1];
                }
                part[(warp * 2 + (tile == first_tile ? 0 : 1)) * 32 + lane] = v;
            }
#pragma unroll
            for (int b = 0; b < NB; ++b) acc[b][0] = acc[b][1] = 0.f;
            k = 0;
            ++tile;
            if (SEL && M.xsel) xcol = tile / M.etiles;
        }
    };
    long long wait_cyc = 0;
    const long long loop_t0 = clock64();
#pragma unroll 1
    for (int u = u0; u < u1;) {
        const int n = min(kSlotUnits, u1 - u);   // the units of this slot (as issued)
        if (tr != nullptr) {
            const long long c0 = clock64();
            ring_wait(r, p, r.consumed);
            wait_cyc += clock64() - c0;
        } else {
            ring_wait(r, p, r.consumed);
        }
        __syncwarp();
        const unsigned char* sg = ring_g + (size_t)(r.consumed % kStages) * kSlotBytes;
#pragma unroll 1
        for (int i = 0; i < n; ++i) {
            unit(sg + i * kUnitBytes, k);
            advance(u + i);
        }
        __syncwarp();
        ++r.consumed;
        ring_issue<W, SEL>(r, mats, warp, lane);   // refill the slot just read
        u += n;
    }
    ring = r;
    stamp(tr, 3);
    if (tr != nullptr && threadIdx.x == 0) {   // warp 0: cycles waiting for ring slots / in the loop
        tr[6] = (unsigned long long)wait_cyc;
        tr[7] = (unsigned long long)(clock64() - loop_t0);
    }
    __syncthreads();
    stamp(tr, 4);
    // A tile shared by several warps is finished by the warp holding its last unit: the sums
    // of every warp that touched it, added in warp order.
    if (u1 > u0) {
        const int ts = (first_tile - T0) * nst;
        if (u0 > ts && u1 >= ts + nst) {
            float s2[NB][2];
#pragma unroll
            for (int b = 0; b < NB; ++b) s2[b][0] = s2[b][1] = 0.f;
            for (int w2 = 0; w2 <= warp; ++w2) {
                const int a0 = warp_unit<W>(U, w2), a1 = warp_unit<W>(U, w2 + 1);
                if (a1 <= a0 || a1 <= ts || a0 >= ts + nst) continue;
                const int sl = a0 >= ts ? 0 : 1;   // begun in this tile: parked as that warp's first
                const float4 v = part[(w2 * 2 + sl) * 32 + lane];
                s2[0][0] += v.x;
                s2[0][1] += v.y;
                if (NB > 1) {
                    s2[NB > 1 ? 1 : 0][0] += v.z;
                    s2[NB > 1 ? 1 : 0][1] += v.w;
                }
            }
            finish_tile<NB>(p, M, epi, first_tile, s2, y, ld, best, lane);
        }
    }
    if (epi == kEpiLogits) {
#pragma unroll
        for (int b = 0; b < NB; ++b) {
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long k2 = __shfl_xor_sync(0xffffffffu, best[b], o);
                best[b] = k2 > best[b] ? k2 : best[b];
            }
            if (lane == 0) kred[warp][b] = best[b];
        }
        __syncthreads();
        if (tid < NB) {
            unsigned long long m = 0ull;
#pragma unroll
            for (int i = 0; i < W; ++i) m = kred[i][tid] > m ? kred[i][tid] : m;
            const bool act = p.active == nullptr || p.active[tid] != 0;
            if (m && act) atomicMax(p.keys + tid, m);
        }
    }
    if (tr != nullptr) __syncthreads();   // the stamp marks the end of every warp's epilogue
    stamp(tr, 5);
}

// ------------------------------------------------------------------------------ attention
// RMSNorm over one head (weight w) and NeoX rotation with the table rows of the position, by
// one warp: lane handles the pairs (i, i + HD/2), i = lane, lane + 32, ...; writes f16 to dst.
template <int HD>
__device__ __forceinline__ void norm_rope(const float* src, const float* w, const float* cr, const float* sr,
                                          float eps, __half* dst, int lane) {
    constexpr int H2 = HD / 2, PER = H2 / 32;
    float xa[PER], xb[PER];
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        xa[k] = __ldcg(src + lane + 32 * k);
        xb[k] = __ldcg(src + lane + 32 * k + H2);
        ss += xa[k] * xa[k] + xb[k] * xb[k];
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = rsqrtf(fmaf(ss, 1.0f / (float)HD, eps));
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int i = lane + 32 * k;
        const float a = xa[k] * r * w[i], bb = xb[k] * r * w[i + H2];
        const float c = cr[i], sn = sr[i];
        dst[i] = __float2half_rn(a * c - bb * sn);
        dst[i + H2] = __float2half_rn(a * sn + bb * c);
    }
}

template <int DPL> struct VRow;
template <> struct VRow<2> {
    using T = unsigned int;
    static __device__ __forceinline__ void f(T u, float (&v)[2]) {
        const float2 a = __half22float2(as_h2(u));
        v[0] = a.x; v[1] = a.y;
    }
};
template <> struct VRow<4> {
    using T = uint2;
    static __device__ __forceinline__ void f(T u, float (&v)[4]) {
        const float2 a = __half22float2(as_h2(u.x)), b = __half22float2(as_h2(u.y));
        v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
    }
};

// Attention of one layer for every (sequence, kv head, split) item; item i runs on CTA
// i mod gridDim.x. Splits: the sequence's blocks are cut into nsplit ranges of spb blocks; the
// range holding the newest position also normalises, rotates and appends the new K/V. Each warp
// issues the loads of its first block before anything else (the new row, not yet in the pool
// then, is patched in from shared memory), so the K/V latency overlaps the q normalisation.
template <int HD, int G>
__device__ __noinline__ void attn_phase(const PersistParams& p, int layer, unsigned char* region,
                                        __half (*qs)[HD], int* flag, unsigned long long* tr) {
    constexpr int NCH = HD / 32;   // 32-dim chunks of a K row (one 16-byte load per lane each)
    constexpr int DPL = HD / 32;   // P.V output dims per lane
    constexpr int WST = G * HD > 128 ? G * HD : 128;   // floats per warp in the merge buffer
    constexpr int ITEMS = G * HD / 4;                   // float4 outputs of a split merge
    constexpr int TPI = kT / ITEMS;                     // threads per output in the split merge
    static_assert(TPI >= 1 && TPI <= 32 && (TPI & (TPI - 1)) == 0, "split merge layout");
    using VT = typename VRow<DPL>::T;
    __shared__ __align__(16) __half knew[HD];   // the appended K row (normed, rotated) and V row
    __shared__ __align__(16) __half vnew[HD];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    float* wacc = reinterpret_cast<float*>(region);   // [kW][WST] (first [G][16]: probabilities)
    float* wm = wacc + kW * WST;                        // [kW][G]
    float* wl = wm + kW * G;
    const PLayer& Ly = p.layers[layer];
    const size_t lp = (size_t)layer * p.layer_pool;
    __half* kpool = p.k_pool + lp;
    __half* vpool = p.v_pool + lp;
    const int nitems = p.B * p.nkv * p.nsplit;
    const size_t qkv_ld = (size_t)(p.nh + 2 * p.nkv) * HD;

    for (int item = blockIdx.x; item < nitems; item += gridDim.x) {
        const int s = item % p.nsplit, bk = item / p.nsplit, kvh = bk % p.nkv, b = bk / p.nkv;
        if (p.active && p.active[b] == 0) continue;
        const int pos = p.positions[b];
        const int L = pos + 1;
        if (pos < 0 || L > p.maxb * kBS || pos >= p.max_position) {
            if (s == 0 && kvh == 0 && tid == 0) record_device_error(p.err, kErrAttnLength, b, L);
            continue;
        }
        const int nblocks = (L + kBS - 1) / kBS;
        const int spb = (nblocks + p.nsplit - 1) / p.nsplit;
        const int n_active = (nblocks + spb - 1) / spb;
        if (s >= n_active) continue;
        const int blk0 = s * spb, blk1 = min(nblocks, blk0 + spb);
        const int lblk = pos / kBS, kp = pos % kBS;
        const int32_t* bt = p.block_tables + (size_t)b * p.maxb;
        __syncthreads();   // the previous item's readers of qs, knew/vnew and the merge buffers are done

        // K/V of block blk straight into registers: K as MMA B fragments (key g and g + 8 of
        // the block, head_dim permuted: lane t of chunk m holds dims 32 m + 8 t .. + 7), V rows
        // as DPL dims per lane; false (error recorded) if the table entry is out of range
        uint4 k0[NCH], k1[NCH];
        VT vv[kBS];
        auto load_block = [&](int blk) -> bool {
            const int phys = bt[blk];
            if (phys < 0 || phys >= p.num_blocks) {
                if (lane == 0) record_device_error(p.err, kErrAttnBlock, (long long)b * p.maxb + blk, phys);
                return false;
            }
            const __half* kb = kpool + ((size_t)phys * p.nkv + kvh) * kBS * HD;
            const __half* vb = vpool + ((size_t)phys * p.nkv + kvh) * kBS * HD;
            const int nt = min(kBS, L - blk * kBS);
#pragma unroll
            for (int m = 0; m < NCH; ++m) {
                k0[m] = __ldcg(reinterpret_cast<const uint4*>(kb + (size_t)g * HD + 32 * m + 8 * t));
                k1[m] = __ldcg(reinterpret_cast<const uint4*>(kb + (size_t)(g + 8) * HD + 32 * m + 8 * t));
            }
#pragma unroll
            for (int kk = 0; kk < kBS; ++kk)
                if (kk < nt) vv[kk] = __ldcg(reinterpret_cast<const VT*>(vb + (size_t)kk * HD + lane * DPL));
            return true;
        };
        bool okA = blk0 + warp < blk1 ? load_block(blk0 + warp) : false;

        const float* src = p.qkv + (size_t)b * qkv_ld;
        const float* cr = p.cos_t + (size_t)pos * (HD / 2);
        const float* sr = p.sin_t + (size_t)pos * (HD / 2);
        if (warp < G) norm_rope<HD>(src + (size_t)(kvh * G + warp) * HD, Ly.q_norm, cr, sr, p.eps, qs[warp], lane);
        if (lblk >= blk0 && lblk < blk1 && warp >= kW - 2) {
            const int phys = bt[lblk];
            if (phys < 0 || phys >= p.num_blocks) {
                if (lane == 0 && warp == kW - 1)
                    record_device_error(p.err, kErrRopeBlock, (long long)b * p.maxb + lblk, phys);
            } else {
                const size_t off = (((size_t)phys * p.nkv + kvh) * kBS + kp) * HD;
                if (warp == kW - 1) {
                    norm_rope<HD>(src + (size_t)(p.nh + kvh) * HD, Ly.k_norm, cr, sr, p.eps, knew, lane);
                    __syncwarp();
                    for (int i = lane; i < HD / 8; i += 32)
                        reinterpret_cast<uint4*>(kpool + off)[i] = reinterpret_cast<const uint4*>(knew)[i];
                } else {
                    const float* vs = src + (size_t)(p.nh + p.nkv + kvh) * HD;
                    for (int i = lane; i < HD; i += 32) {
                        const __half v = __float2half_rn(__ldcg(vs + i));
                        vnew[i] = v;
                        vpool[off + i] = v;
                    }
                }
            }
        }
        __syncthreads();   // qs, knew and vnew are complete
        stamp(tr, 2);

        // Q as the A operand of S = Q K^T (rows = the G heads, rows >= G zero), permuted like K
        uint4 qf[NCH];
#pragma unroll
        for (int m = 0; m < NCH; ++m)
            qf[m] = g < G ? *reinterpret_cast<const uint4*>(&qs[g][32 * m + 8 * t]) : make_uint4(0u, 0u, 0u, 0u);
        float o[G][DPL];
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int d = 0; d < DPL; ++d) o[h][d] = 0.f;
        float mrun = -INFINITY, lrun = 0.f;   // running max / sum of head g (lanes g < G)
        float* pb = wacc + warp * WST;
        bool any = false;
        for (int blk = blk0 + warp, i = 0; blk < blk1; blk += kW, ++i) {
            const bool ok = i == 0 ? okA : load_block(blk);
            if (!ok) continue;
            any = true;
            const int nt = min(kBS, L - blk * kBS);   // valid keys of the block
            if (blk == lblk) {   // the appended row (its pool copy may postdate the loads above)
#pragma unroll
                for (int m = 0; m < NCH; ++m) {
                    if (g == kp) k0[m] = *reinterpret_cast<const uint4*>(&knew[32 * m + 8 * t]);
                    if (g + 8 == kp) k1[m] = *reinterpret_cast<const uint4*>(&knew[32 * m + 8 * t]);
                }
#pragma unroll
                for (int kk = 0; kk < kBS; ++kk)
                    if (kk == kp) vv[kk] = *reinterpret_cast<const VT*>(&vnew[lane * DPL]);
            }
            float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int m = 0; m < NCH; ++m) {
                mma16816(s0, qf[m].x, 0u, qf[m].y, 0u, k0[m].x, k0[m].y);
                mma16816(s0, qf[m].z, 0u, qf[m].w, 0u, k0[m].z, k0[m].w);
                mma16816(s1, qf[m].x, 0u, qf[m].y, 0u, k1[m].x, k1[m].y);
                mma16816(s1, qf[m].z, 0u, qf[m].w, 0u, k1[m].z, k1[m].w);
            }
            // online softmax of head row g over keys 2t, 2t + 1, 2t + 8, 2t + 9 (exp2 domain);
            // keys past the context are excluded by selection (their K rows may be garbage)
            const int c0 = 2 * t;
            const float x0 = c0 < nt ? s0[0] * p.scale_log2 : -INFINITY;
            const float x1 = c0 + 1 < nt ? s0[1] * p.scale_log2 : -INFINITY;
            const float x2 = c0 + 8 < nt ? s1[0] * p.scale_log2 : -INFINITY;
            const float x3 = c0 + 9 < nt ? s1[1] * p.scale_log2 : -INFINITY;
            float mb = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
            mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
            mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
            const float mn = fmaxf(mrun, mb);   // finite: key 0 of the block is valid
            const float alpha = exp2f(mrun - mn);
            const float e0 = exp2f(x0 - mn), e1 = exp2f(x1 - mn), e2 = exp2f(x2 - mn), e3 = exp2f(x3 - mn);
            float ls = (e0 + e1) + (e2 + e3);
            ls += __shfl_xor_sync(0xffffffffu, ls, 1);
            ls += __shfl_xor_sync(0xffffffffu, ls, 2);
            lrun = lrun * alpha + ls;
            mrun = mn;
            if (g < G) {
                pb[g * 16 + c0] = e0;
                pb[g * 16 + c0 + 1] = e1;
                pb[g * 16 + c0 + 8] = e2;
                pb[g * 16 + c0 + 9] = e3;
            }
            __syncwarp();
            // O = alpha O + P V: lane owns dims DPL * lane .. + DPL - 1 of every head
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float ah = __shfl_sync(0xffffffffu, alpha, 4 * h);
#pragma unroll
                for (int d = 0; d < DPL; ++d) o[h][d] *= ah;
            }
#pragma unroll
            for (int kk = 0; kk < kBS; ++kk) {
                if (kk < nt) {
                    float v[DPL];
                    VRow<DPL>::f(vv[kk], v);
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const float pv = pb[h * 16 + kk];
#pragma unroll
                        for (int d = 0; d < DPL; ++d) o[h][d] = fmaf(pv, v[d], o[h][d]);
                    }
                }
            }
            __syncwarp();
        }
        // this warp's state: lane 4h holds (m, l) of head h; every lane its dims of every head
        if (any) {
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int d = 0; d < DPL; ++d) pb[h * HD + DPL * lane + d] = o[h][d];
            if (t == 0 && g < G) {
                wm[warp * G + g] = mrun;
                wl[warp * G + g] = lrun;
            }
        } else if (lane < G) {
            wm[warp * G + lane] = -INFINITY;
            wl[warp * G + lane] = 0.f;
        }
        __syncthreads();
        stamp(tr, 3);
        for (int i = tid; i < G * HD; i += kT) {
            const int h = i / HD, d = i - h * HD;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kW; ++w) M = fmaxf(M, wm[w * G + h]);
            float Ls = 0.f, A = 0.f;
#pragma unroll
            for (int w = 0; w < kW; ++w) {
                const float mw = wm[w * G + h];
                if (mw != -INFINITY) {
                    const float f = exp2f(mw - M);
                    Ls += wl[w * G + h] * f;
                    A += wacc[w * WST + h * HD + d] * f;
                }
            }
            const int hg = kvh * G + h;
            if (n_active == 1) {
                p.attn[((size_t)b * p.nh + hg) * HD + d] = __float2half_rn(A / Ls);
            } else {
                const size_t slot = ((size_t)b * p.nh + hg) * p.nsplit + s;
                p.pacc[slot * HD + d] = A;
                if (d == 0) {
                    p.pm[slot] = M;
                    p.pl[slot] = Ls;
                }
            }
        }
        if (n_active == 1) continue;

        // split merge in the CTA that arrives last (no waiting): an acq_rel ticket publishes
        // this CTA's partials (ordered before it by the bar.sync) and, for the last CTA, makes
        // every other CTA's partials visible
        __syncthreads();
        if (tid == 0) {
            unsigned int old;
            asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                         : "=r"(old)
                         : "l"(p.tickets + b * p.nkv + kvh)
                         : "memory");
            *flag = (int)old == n_active - 1;
        }
        __syncthreads();
        stamp(tr, 4);
        if (!*flag) continue;
        // TPI threads per float4 output, each over splits sub, sub + TPI, ... (online softmax),
        // all loads of a thread issued together; the TPI states are then combined by shuffles
        {
            const int it = tid / TPI, sub = tid % TPI;
            const int h = it / (HD / 4), d4 = it - h * (HD / 4);
            const size_t base = ((size_t)b * p.nh + kvh * G + h) * p.nsplit;
            const float4* srcp = reinterpret_cast<const float4*>(p.pacc) + base * (HD / 4) + d4;
            float M = -INFINITY, Ls = 0.f;
            float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int k0s = sub; k0s < n_active; k0s += 4 * TPI) {
                float mk[4], lk[4];
                float4 ak[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int k = k0s + u * TPI;
                    if (k < n_active) {
                        mk[u] = __ldcg(p.pm + base + k);
                        lk[u] = __ldcg(p.pl + base + k);
                        ak[u] = __ldcg(srcp + (size_t)k * (HD / 4));
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int k = k0s + u * TPI;
                    if (k < n_active && mk[u] != -INFINITY) {
                        const float mn = fmaxf(M, mk[u]);
                        const float fo = exp2f(M - mn), fk = exp2f(mk[u] - mn);
                        Ls = Ls * fo + lk[u] * fk;
                        A.x = A.x * fo + ak[u].x * fk; A.y = A.y * fo + ak[u].y * fk;
                        A.z = A.z * fo + ak[u].z * fk; A.w = A.w * fo + ak[u].w * fk;
                        M = mn;
                    }
                }
            }
#pragma unroll
            for (int o2 = 1; o2 < TPI; o2 <<= 1) {
                const float Mo = __shfl_xor_sync(0xffffffffu, M, o2);
                const float Lo = __shfl_xor_sync(0xffffffffu, Ls, o2);
                float4 Ao;
                Ao.x = __shfl_xor_sync(0xffffffffu, A.x, o2);
                Ao.y = __shfl_xor_sync(0xffffffffu, A.y, o2);
                Ao.z = __shfl_xor_sync(0xffffffffu, A.z, o2);
                Ao.w = __shfl_xor_sync(0xffffffffu, A.w, o2);
                const float mn = fmaxf(M, Mo);
                if (mn != -INFINITY) {
                    const float fa = exp2f(M - mn), fb = exp2f(Mo - mn);
                    Ls = Ls * fa + Lo * fb;
                    A.x = A.x * fa + Ao.x * fb; A.y = A.y * fa + Ao.y * fb;
                    A.z = A.z * fa + Ao.z * fb; A.w = A.w * fa + Ao.w * fb;
                    M = mn;
                }
            }
            if (sub == 0) {
                const float inv = 1.0f / Ls;
                __half* out = p.attn + ((size_t)b * p.nh + kvh * G + h) * HD + d4 * 4;
                *reinterpret_cast<__half2*>(out) = __floats2half2_rn(A.x * inv, A.y * inv);
                *reinterpret_cast<__half2*>(out + 2) = __floats2half2_rn(A.z * inv, A.w * inv);
            }
        }
        if (tid == 0) p.tickets[b * p.nkv + kvh] = 0;   // re-arm for the next layer / step
        stamp(tr, 5);
    }
}

// ------------------------------------------------------------------------------ the step
// x[b] = E[token[b]] (f32 residual stream), split evenly over the CTAs.
static __device__ void embed_phase(const PersistParams& p) {
    const int n4 = p.hidden / 4;
    const long long total = (long long)p.B * n4;
    const long long i0 = (long long)blockIdx.x * total / gridDim.x;
    const long long i1 = (long long)(blockIdx.x + 1) * total / gridDim.x;
    for (long long i = i0 + threadIdx.x; i < i1; i += kT) {
        const int b = (int)(i / n4), c = (int)(i - (long long)b * n4);
        int tok = p.tokens[b];
        if (tok < 0 || tok >= p.vocab) {
            if (c == 0 && (p.active == nullptr || p.active[b] != 0))
                record_device_error(p.err, kErrEmbedToken, b, tok);
            tok = 0;
        }
        reinterpret_cast<float4*>(p.x)[i] = __ldg(reinterpret_cast<const float4*>(p.embed + (size_t)tok * p.hidden) + c);
    }
}

// Next token (argmax key), position + 1, keys re-armed; CTA 0 after the last barrier.
static __device__ void finalize(const PersistParams& p) {
    const int b = threadIdx.x;
    if (b >= p.B) return;
    const unsigned long long k = atomicExch(p.keys + b, 0ull);
    if (p.active && p.active[b] == 0) return;
    const int tok = (int)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull));
    const int pos = p.positions[b];
    p.next_tokens[b] = tok;
    if (p.out_tokens && pos + 1 >= 0 && pos + 1 < p.out_stride)
        p.out_tokens[(size_t)b * p.out_stride + pos + 1] = tok;
    p.positions[b] = pos + 1;
}

// Ask L2 for the K/V tiles this CTA's attention items of `layer` will read (a hint: issued at
// the start of the layer's q|k|v phase, so that the attention phase finds them in L2).
template <int HD>
__device__ void attn_prefetch(const PersistParams& p, int layer) {
    const int nitems = p.B * p.nkv * p.nsplit;
    const size_t lp = (size_t)layer * p.layer_pool;
    for (int item = blockIdx.x; item < nitems; item += gridDim.x) {
        const int s = item % p.nsplit, bk = item / p.nsplit, kvh = bk % p.nkv, b = bk / p.nkv;
        if (p.active && p.active[b] == 0) continue;
        const int L = p.positions[b] + 1;
        if (L <= 0 || L > p.maxb * kBS) continue;
        const int nblocks = (L + kBS - 1) / kBS;
        const int spb = (nblocks + p.nsplit - 1) / p.nsplit;
        const int blk0 = s * spb, blk1 = min(nblocks, blk0 + spb);
        for (int i = threadIdx.x; i < 2 * (blk1 - blk0); i += kT) {
            const int phys = p.block_tables[(size_t)b * p.maxb + blk0 + (i >> 1)];
            if (phys < 0 || phys >= p.num_blocks) continue;
            const __half* base = ((i & 1) ? p.v_pool : p.k_pool) + lp + ((size_t)phys * p.nkv + kvh) * kBS * HD;
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(base), "r"((uint32_t)(kBS * HD * 2))
                         : "memory");
        }
    }
}

template <int HD, int G, int NB>
__device__ void step_body(const PersistParams& p, const PMat* mats, Ring& r, unsigned char* region, __half (*qs)[HD],
                          unsigned long long (*kred)[kMaxB], int* flag) {
    const Hot hot{p.B, p.max_nblk, p.eps};
    unsigned int target = 0;
    // trace row of the barrier that ends the next phase
    auto row = [&]() -> unsigned long long* {
        return p.trace ? p.trace + ((size_t)(target / gridDim.x + 1) * gridDim.x + blockIdx.x) * kTraceWords : nullptr;
    };
    embed_phase(p);
    if (!grid_barrier(p, target, flag)) return;
    const int qkv_ld = (p.nh + 2 * p.nkv) * HD;
    for (int l = 0; l < p.n_layers; ++l) {
        const PLayer* Ly = p.layers + l;
        attn_prefetch<HD>(p, l);
        // q|k|v = W_qkv rmsnorm(x, attn_norm)
        gemv_phase<NB, kW>(p, hot, mats, 4 * l, kEpiF32, true, r, p.x, nullptr, Ly->attn_norm, p.qkv, qkv_ld, region,
                                      kred, row());
        if (!grid_barrier(p, target, flag)) return;
        // qk-norm + RoPE + KV append + paged attention -> attn
        attn_phase<HD, G>(p, l, region, qs, flag, row());
        if (!grid_barrier(p, target, flag)) return;
        // x += W_o attn
        gemv_phase<NB, kW>(p, hot, mats, 4 * l + 1, kEpiResid, false, r, nullptr, p.attn, nullptr, p.x, p.hidden, region,
                                         kred, row());
        if (!grid_barrier(p, target, flag)) return;
        // act = silu(gate) * up, [gate | up] = W_gu rmsnorm(x, ffn_norm)
        gemv_phase<NB, kW>(p, hot, mats, 4 * l + 2, kEpiSilu, true, r, p.x, nullptr, Ly->ffn_norm, p.act, p.inter, region,
                                       kred, row());
        if (!grid_barrier(p, target, flag)) return;
        // x += W_down act
        gemv_phase<NB, kW>(p, hot, mats, 4 * l + 3, kEpiResid, false, r, nullptr, p.act, nullptr, p.x, p.hidden, region,
                                         kred, row());
        if (!grid_barrier(p, target, flag)) return;
    }
    // logits = W_lm rmsnorm(x, final_norm), greedy argmax keys
    gemv_phase<NB, kW>(p, hot, mats, 4 * p.n_layers, kEpiLogits, true, r, p.x, nullptr, p.final_norm, p.logits, p.vocab, region,
                                     kred, row());
    if (!grid_barrier(p, target, flag)) return;
    if (blockIdx.x == 0) finalize(p);
}

// Dynamic shared memory: [weight rings][GEMV staging | attention merge][matrix descriptors].
__host__ __device__ constexpr size_t region_bytes(int batch, int max_nblk, int head_dim, int group) {
    return gemv_region_bytes(batch, max_nblk) > attn_region_bytes(head_dim, group) ? gemv_region_bytes(batch, max_nblk)
                                                                                   : attn_region_bytes(head_dim, group);
}

template <int HD, int G>
__global__ void __launch_bounds__(kT, 1) step_kernel(const __grid_constant__ PersistParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ __align__(16) __half qs[G][HD];
    __shared__ unsigned long long kred[kW][kMaxB];
    __shared__ int flag;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned char* region = smem + kRingBytes;
    PMat* mats = reinterpret_cast<PMat*>(region + region_bytes(p.B, p.max_nblk, HD, G));
    if (p.trace && threadIdx.x == 0)
        p.trace[kTraceWords * blockIdx.x] = p.trace[kTraceWords * blockIdx.x + 1] = global_ns();
    const int nmat = 4 * p.n_layers + 1;
    for (int i = threadIdx.x; i < nmat; i += kT) mats[i] = mat_global(p, i);
    __syncthreads();
    // per-warp ring slots, one mbarrier each (arrival count 1: the issuing lane)
    __shared__ __align__(8) unsigned long long mbar[kW * kStages];
    if (lane == 0)
        for (int i = 0; i < kStages; ++i)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(
                             static_cast<uint32_t>(__cvta_generic_to_shared(&mbar[warp * kStages + i]))) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();
    Ring r;
    r.wp = 0;
    r.nmat = nmat;
    r.u = r.u_end = 0;
    r.src = nullptr;
    r.issued = r.consumed = 0;
    r.dead = 0;
    r.base = static_cast<uint32_t>(__cvta_generic_to_shared(smem)) + (uint32_t)(warp * kStages * kSlotBytes);
    r.mbar = static_cast<uint32_t>(__cvta_generic_to_shared(&mbar[warp * kStages]));
    ring_seek<kW>(r, mats, warp);
    // the weights do not depend on anything computed in the step: start streaming at once
#pragma unroll 1
    for (int i = 0; i < kStages; ++i) ring_issue<kW>(r, mats, warp, lane);
    if (p.B == 1)
        step_body<HD, G, 1>(p, mats, r, region, qs, kred, &flag);
    else
        step_body<HD, G, 2>(p, mats, r, region, qs, kred, &flag);
    // after an early exit, let this warp's copies still in flight land before leaving (bounded:
    // past the bound the CTA leaves anyway)
    const unsigned long long t0 = global_ns();
    while (r.consumed < r.issued) {
        const uint32_t mb = r.mbar + (r.consumed % kStages) * 8, parity = (r.consumed / kStages) & 1u;
        bool landed = mbar_test(mb, parity);
        while (!landed && global_ns() - t0 <= p.barrier_timeout_ns) landed = mbar_test(mb, parity);
        if (!landed) break;
        ++r.consumed;
    }
    leave_step(p);
}

// ------------------------------------------------------------------------------ stream layout
// Re-lay a q4_0 matrix (codes [rows][nblk][16], f16 scales [rows][nblk]) into the tile stream
// layout, one warp per 1152-byte unit; rows past the matrix are zero (a zero scale: no
// contribution). An exact byte permutation.
static __global__ void stream_pack_kernel(PMat M, uint8_t* out) {
    const int lane = threadIdx.x & 31;
    const int nst = M.nblk / kUnitBlocks;
    const long long nunits = (long long)M.ntile * nst;
    const long long wpb = blockDim.x / 32;
    for (long long u = blockIdx.x * wpb + (threadIdx.x >> 5); u < nunits; u += (long long)gridDim.x * wpb) {
        const int tile = (int)(u / nst), k = (int)(u % nst);
        uint8_t* dst = out + u * kUnitBytes;
        for (int c = lane; c < kUnitBlocks * 16; c += 32) {
            const int q = c >> 4, r = c & 15;
            bool ok;
            const int row = tile_row(M, tile, r, ok);
            const uint4 v = ok ? *reinterpret_cast<const uint4*>(M.quants + ((size_t)row * M.nblk + kUnitBlocks * k + q) * 16)
                               : make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(dst + c * 16) = v;
        }
        if (lane < 16) {
            bool ok;
            const int row = tile_row(M, tile, lane, ok);
            const uint2 v = ok ? *reinterpret_cast<const uint2*>(M.scales + (size_t)row * M.nblk + kUnitBlocks * k)
                               : make_uint2(0u, 0u);
            *reinterpret_cast<uint2*>(dst + kUnitBlocks * 16 * 16 + lane * 8) = v;
        }
    }
}

// ------------------------------------------------------------------------------ stand-alone GEMV
// One GEMV phase as its own kernel (one CTA per SM), for the step that runs one launch per
// phase: the ring's first slots are filled before the kernel waits on its predecessor
// (programmatic dependent launch), since the weights do not depend on it.
struct StreamGemv {
    PMat M;
    int epi, rms;
    const float* xf;       // rms: f32 [B][cols], normalised with norm_w
    const __half* x16;     // else: f16 [B][cols]
    const float* norm_w;
    void* y;
    int ld;
    unsigned long long* trace;   // optional [grid][kTraceWords]: 0 start, 1 after the wait, 2-7 as
                                 // in gemv_phase
    NextWeights next;            // prefetched into L2 before the wait
    int prewait;                 // ring slots issued before the wait (the rest after staging)
};

template <int NB, int W, bool I8, bool SEL = false>
__global__ void __launch_bounds__(W * 32, 16 / W) gemv_stream_kernel(const __grid_constant__ PersistParams p,
                                                                      const __grid_constant__ StreamGemv g) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ PMat mat;
    __shared__ unsigned long long kred[W][kMaxB];
    __shared__ __align__(8) unsigned long long mbar[W * kStages];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long* tr = g.trace ? g.trace + (size_t)blockIdx.x * kTraceWords : nullptr;
    stamp(tr, 0);
    if (threadIdx.x == 0) mat = g.M;
    if (lane == 0)
        for (int i = 0; i < kStages; ++i)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(
                             static_cast<uint32_t>(__cvta_generic_to_shared(&mbar[warp * kStages + i]))) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();
    Ring r;
    r.wp = 0;
    r.nmat = 1;
    r.u = r.u_end = 0;
    r.src = nullptr;
    r.issued = r.consumed = 0;
    r.dead = 0;
    r.base = static_cast<uint32_t>(__cvta_generic_to_shared(smem)) + (uint32_t)(warp * kStages * kSlotBytes);
    r.mbar = static_cast<uint32_t>(__cvta_generic_to_shared(&mbar[warp * kStages]));
    ring_seek<W>(r, &mat, warp);
#pragma unroll 1
    for (int i = 0; i < g.prewait; ++i) ring_issue<W, SEL>(r, &mat, warp, lane);
    // constants of a later kernel of the step (its norm weights), into L2 off its critical path
    l2_prefetch_share(g.next.ptr[0], g.next.bytes[0]);
    l2_prefetch_share(g.next.ptr[1], g.next.bytes[1]);
    const Hot hot = hot_scalars(p);
    // the trigger follows the wait in every kernel of the step: a kernel's code before its
    // wait then runs only after the kernel two launches back has completed
    pdl_wait();
    pdl_trigger();
    stamp(tr, 1);
    gemv_phase<NB, W, I8, SEL>(p, hot, &mat, 0, g.epi, g.rms != 0, r, g.xf, g.x16, g.norm_w, g.y, g.ld,
                               smem + (size_t)W * kStages * kSlotBytes, kred, tr);
    const unsigned long long t0 = global_ns();
    while (r.consumed < r.issued) {   // only after a wait ran out: let copies land (bounded)
        const uint32_t mb = r.mbar + (r.consumed % kStages) * 8, parity = (r.consumed / kStages) & 1u;
        bool landed = mbar_test(mb, parity);
        while (!landed && global_ns() - t0 <= p.barrier_timeout_ns) landed = mbar_test(mb, parity);
        if (!landed) break;
        ++r.consumed;
    }
}

}  // namespace persist
}  // namespace ql

// ------------------------------------------------------------------------------ host side
namespace ql {
namespace persist {

// Set the kernel's attributes and report its occupancy (launch == false), or launch it as a
// cooperative grid of `grid` CTAs (launch == true).
template <int HD, int G>
cudaError_t run_one(bool launch, const PersistParams* p, size_t smem, int grid, cudaStream_t s, int* occ) {
    if (!launch) {
        // allow the device's whole opt-in shared memory (models of other shapes share the kernel),
        // then check that `smem` bytes leave one CTA per SM
        int dev = 0, optin = 0;
        cudaFuncAttributes fa = {};
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, step_kernel<HD, G>);
        if (e == cudaSuccess && smem + fa.sharedSizeBytes > (size_t)optin) {
            *occ = 0;
            return cudaSuccess;
        }
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(step_kernel<HD, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     optin - (int)fa.sharedSizeBytes);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, step_kernel<HD, G>, kT, smem);
        return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, step_kernel<HD, G>, *p);
}

template <int HD>
cudaError_t dispatch(int G, bool launch, const PersistParams* p, size_t smem, int grid, cudaStream_t s, int* occ) {
    switch (G) {
        case 1: return run_one<HD, 1>(launch, p, smem, grid, s, occ);
        case 2: return run_one<HD, 2>(launch, p, smem, grid, s, occ);
        case 4: return run_one<HD, 4>(launch, p, smem, grid, s, occ);
        case 8: return run_one<HD, 8>(launch, p, smem, grid, s, occ);
        default: return cudaErrorInvalidValue;
    }
}

template <typename K, typename... Args>
cudaError_t launch_kernel_pdl(K kernel, int grid, int threads, size_t smem, cudaStream_t s, bool pdl,
                              const Args&... args) {
    return ql::launch(kernel, dim3(grid), dim3(threads), smem, s, pdl, args...);
}

template <int NB, int W, bool I8 = false, bool SEL = false>
cudaError_t stream_gemv_one(bool launch, const PersistParams* p, const StreamGemv* g, size_t smem, int grid,
                            cudaStream_t s, bool pdl) {
    auto* k = gemv_stream_kernel<NB, W, I8, SEL>;
    if (!launch) {
        int dev = 0, optin = 0;
        cudaFuncAttributes fa = {};
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, k);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - (int)fa.sharedSizeBytes);
        return e;
    }
    return launch_kernel_pdl(k, grid, W * 32, smem, s, pdl, *p, *g);
}

}  // namespace persist

// One translation unit per head_dim (they compile in parallel).
cudaError_t persist_dispatch_hd64(int G, bool launch, const PersistParams* p, size_t smem, int grid,
                                  cudaStream_t s, int* occ);
cudaError_t persist_dispatch_hd128(int G, bool launch, const PersistParams* p, size_t smem, int grid,
                                   cudaStream_t s, int* occ);

}  // namespace ql
