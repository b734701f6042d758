// q4_0 GEMM for prompt chunks: y[t][r] = sum_k W[r][k] x[t][k] for a chunk of T tokens, on the
// 5th-generation tensor cores (tcgen05) with the weights dequantised on the fly.
//
// [IL] inferencelayer cuda_llm.rs: the module doc runs a prompt as sequential decode, and its
// prefill arm multiplies bf16 copies of the weights with cuBLAS GemmEx. Here the chunk's tokens
// are the N dimension of one GEMM per projection against the same q4_0 tile stream copy of the
// weights that the decode step streams, so every weight byte is read once per 128 tokens and
// no f16 copy of the weights exists: (q - 8) d is formed in registers and stored into tensor
// memory as the MMA's A operand.
//
// One CTA per (block of 128 weight rows = 8 tiles, tile of NT tokens: 256 when the chunk has
// more than 128 tokens, 128 when it has more than 32, else 32); K streams in units of 128
// columns (one 1152-byte unit of each tile):
//  * warp 17, lane 0: per unit, one tensor-map copy of the row block's 8 tiles x 1 unit of codes
//    and scales (tiles past the matrix read as zero) into a ring of kSW stages. The first kSW
//    go out before the wait on the previous kernel (the weights do not depend on it);
//  * warp 18, lane 0: per unit, two tensor-map copies of the tokens' activations (64 f16 of K x
//    NT tokens each: each token's 128 bytes one row, with the 128-byte swizzle, i.e. the K-major
//    layout the MMA reads with a SWIZZLE_128B descriptor; tokens past the chunk read as zero)
//    into a ring of kSB stages (kSW and kSB by NT, as many as the shared memory holds);
//  * warps 0-15 (warp w serves tensor-memory lanes 32 (w % 4).., i.e. rows 32 (w % 4).. of the
//    block, and the unit's block w / 4): each thread expands its row's 32 codes of that block
//    into (q - 8) d in f16, in K order (two consecutive K per 32-bit column), frees the code
//    stage, and stores the values into one of kA A slots of tensor memory; after the last unit
//    these warps run the epilogue;
//  * warp 16 allocates the tensor memory; its lane 0 issues tcgen05.mma (kind::f16, M 128,
//    N NT, K 16, A in tensor memory, B in shared memory) into one f32 accumulator of NT columns
//    and commits each unit's MMAs to the barriers that free its activation stage and A slot;
//  * epilogue: tcgen05.ld of the accumulator (warp w: its lanes' rows, tokens NT / 4 (w / 4)..),
//    then the stores: f32, added to the residual, or SiLU(gate) * up in f16 (the gate row's
//    thread takes the up row from the lane 8 above).
// The codes (from HBM) and the activations (from L2) have rings of their own, so that the
// codes can run up to kSW units ahead. A matrix with few row blocks is split over K as well
// (blockIdx.z takes a run of units): each CTA then stores its raw f32 sums, and gemm_merge_kernel
// adds the K parts in order and applies the epilogue.
// Every barrier has one waiter role, which takes its phases in order. Every wait is bounded: an
// expiry records a device error and stops the CTA, whose copies in flight land (bounded) and
// whose tensor memory is freed before it leaves.
#include "ql_batched.h"
#include "ql_persist.cuh"

#include <cuda.h>

#include <mutex>
#include <set>

namespace ql {
namespace gemm {

using persist::as_h2;
using persist::as_u32;

constexpr int kUnitBytes = persist::kUnitBytes;   // 16 rows x 128 columns: codes, then scales
constexpr int kRB = 8;                             // tiles per row block: the MMA's M of 128 rows
constexpr int kCodeBytes = kRB * kUnitBytes;       // 9216
constexpr uint32_t kTmemCols = 512;
constexpr int kDW = 16;                            // dequantisation (and epilogue) warps
constexpr int kMmaWarp = kDW, kWProdWarp = kDW + 1, kBProdWarp = kDW + 2, kThreads = (kDW + 3) * 32;

template <int NT>
struct Cfg {
    static constexpr int kSW = NT == 32 ? 4 : 3;                    // code stages (one unit each)
    // units in flight between the dequantisation and the MMAs: unit u's activations (stage
    // u % kSB) and its expanded weights (A slot u % kSB of tensor memory, 64 columns) are freed
    // together by one commit, so the stages and the slots are one ring
    static constexpr int kSB = NT == 256 ? 3 : NT == 128 ? 6 : 7;
    static constexpr int kA = kSB;
    // kReady[s]: unit u's activations landed (the copies' bytes and the producer's arrival) and
    // its A slot stored (one arrival per dequantisation warp): the MMA lane's one wait per unit
    static constexpr int kWFull = 0, kWEmpty = kSW, kReady = 2 * kSW, kFree = 2 * kSW + kSB,
                         kDFull = kFree + kSB, kDone = kDFull + 1, kBars = kDone + 1;
    static constexpr int kBHalf = NT * 128;                // 64 K for NT tokens: one 128-byte-swizzled box
    static constexpr int kBStage = 2 * kBHalf;             // a unit (128 K) for NT tokens
    static constexpr size_t kSmem = (size_t)kSW * kCodeBytes + (size_t)kSB * kBStage;
    static constexpr uint32_t kACol = NT;                  // the A slots after the accumulator's columns
    // instruction descriptor: D f32, A and B f16, both K-major, N = NT, M = 128
    static constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(NT >> 3) << 17) | ((128u >> 4) << 24);
    static_assert(NT + kA * 64 <= (int)kTmemCols, "tensor memory: accumulator + A slots");
    static_assert((kSW * kCodeBytes) % 1024 == 0, "activation stages 1024-byte aligned");
};

struct Params {
    CUtensorMap tw;       // weights: [tile][unit][144 x 8 B], boxes of 8 tiles x 1 unit
    CUtensorMap tx;       // activations: [T][K] f16, boxes of NT tokens x 64, 128-byte swizzle
    int T, rows, nst, silu, epi, ld;
    void* y;
    DevError* err;
    unsigned long long timeout_ns;
    int kparts, upp;      // K parts (blockIdx.z) and units per part
    float* part;          // kparts > 1: [kparts][T][ntile * 16] raw f32 sums (the stream's row order)
    int R;                // ntile * 16
};

__device__ __forceinline__ uint32_t su32(const void* q) { return static_cast<uint32_t>(__cvta_generic_to_shared(q)); }

// Phase `parity` of an mbarrier, bounded: false when the bound runs out (the error recorded, the
// CTA's abort flag raised) or when another role has aborted. abort_flag null: the bound alone.
__device__ __forceinline__ bool wait_bar(uint32_t mb, uint32_t parity, const Params& p, int* abort_flag, int where) {
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
    if (abort_flag == nullptr || atomicExch(abort_flag, 1) == 0)
        record_device_error(p.err, kErrGemvStage, blockIdx.x, where);
    return false;
}

// wait_bar by every lane, one answer for the warp (its collective instructions that follow need
// every lane or none)
__device__ __forceinline__ bool warp_wait(uint32_t mb, uint32_t parity, const Params& p, int* abort_flag, int where) {
    const bool ok = wait_bar(mb, parity, p, abort_flag, where);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void arrive(uint32_t mb) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mb) : "memory");
}

__device__ __forceinline__ void expect_tx(uint32_t mb, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mb), "r"(bytes) : "memory");
}

__device__ __forceinline__ void commit(uint32_t mb) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mb) : "memory");
}

// (q - 8) d of two consecutive codes (nibbles 0-3 of the two 16-bit halves of w), in f16: 1024 + q
// exactly by the exponent trick, less 1032 exactly, times d (one rounding)
__device__ __forceinline__ uint32_t deq2(uint32_t w, __half2 d2) {
    const __half2 off = as_h2(0x64086408u);   // 1032
    return as_u32(__hmul2(__hsub2(as_h2((w & 0x000F000Fu) | 0x64006400u), off), d2));
}

template <int NT>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ Params p) {
    using C = Cfg<NT>;
    constexpr int kSW = C::kSW, kSB = C::kSB, kA = C::kA;
    constexpr int kWFull = C::kWFull, kWEmpty = C::kWEmpty, kReady = C::kReady, kFree = C::kFree,
                  kDFull = C::kDFull, kDone = C::kDone, kBars = C::kBars;
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ __align__(8) unsigned long long bars[kBars];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ int issued_w, issued_b;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rb = blockIdx.x, n0 = blockIdx.y * NT, kp = blockIdx.z;
    const int u0 = kp * p.upp;                         // this CTA's first unit (of the matrix's K)
    const int nst = p.nst - u0 < p.upp ? p.nst - u0 : p.upp;   // its units
    const uint32_t bar = su32(bars);
    unsigned char* bsm = smem + (size_t)kSW * kCodeBytes;   // the activation stages
    if (threadIdx.x == 0) {
        for (int s = 0; s < kSW; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar + (kWFull + s) * 8) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar + (kWEmpty + s) * 8), "r"(kDW) : "memory");
        }
        for (int s = 0; s < kSB; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar + (kReady + s) * 8), "r"(kDW + 1) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar + (kFree + s) * 8) : "memory");
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar + kDFull * 8) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar + kDone * 8) : "memory");
        abort_flag = 0;
        issued_w = issued_b = 0;
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

    const int prew = nst < kSW ? nst : kSW;
    unsigned long long pol = 0;
    auto copy_w = [&](int u) {   // the codes of unit u into stage u % kSW
        const int s = u % kSW;
        expect_tx(bar + (kWFull + s) * 8, (uint32_t)kCodeBytes);
        asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
                     " [%0], [%1, {%2, %3, %4}], [%5], %6;"
                     ::"r"(su32(smem + (size_t)s * kCodeBytes)), "l"(reinterpret_cast<uint64_t>(&p.tw)), "r"(0),
                       "r"(u0 + u), "r"(rb * kRB), "r"(bar + (kWFull + s) * 8), "l"(pol) : "memory");
    };
    if (warp == kWProdWarp && lane == 0) {
        pol = l2_evict_first();
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tw)) : "memory");
        for (int u = 0; u < prew; ++u) copy_w(u);   // before the wait
    }
    if (warp == kBProdWarp && lane == 0)
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tx)) : "memory");
    pdl_wait();
    pdl_trigger();

    if (warp == kWProdWarp) {
        // ------------------------------------------------ code copies (one lane)
        if (lane == 0) {
            int u = prew;
            for (; u < nst; ++u) {
                const int s = u % kSW;
                if (!wait_bar(bar + (kWEmpty + s) * 8, (uint32_t)(u / kSW - 1) & 1u, p, abt, 100 + u)) break;
                // the stage was read through the generic proxy; the copy writes it through the
                // async proxy
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                copy_w(u);
            }
            issued_w = u;
        }
        __syncwarp();
    } else if (warp == kBProdWarp) {
        // ------------------------------------------------ activation copies (one lane)
        if (lane == 0) {
            int u = 0;
            for (; u < nst; ++u) {
                const int s = u % kSB;
                if (u >= kSB && !wait_bar(bar + (kFree + s) * 8, (uint32_t)(u / kSB - 1) & 1u, p, abt, 200 + u)) break;
                expect_tx(bar + (kReady + s) * 8, (uint32_t)C::kBStage);
                for (int hh = 0; hh < 2; ++hh)   // the unit's two 64-K halves
                    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                                 " [%0], [%1, {%2, %3}], [%4];"
                                 ::"r"(su32(bsm + (size_t)s * C::kBStage + (size_t)hh * C::kBHalf)),
                                   "l"(reinterpret_cast<uint64_t>(&p.tx)), "r"(128 * (u0 + u) + 64 * hh), "r"(n0),
                                   "r"(bar + (kReady + s) * 8) : "memory");
            }
            issued_b = u;
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------ MMA issue (one lane)
        if (lane == 0) {
            const uint32_t b0 = su32(bsm);
            for (int u = 0; u < nst; ++u) {
                const int a = u % kA;
                const int s = u % kSB;
                // one wait (the A slot and the activations), one fence, 8 MMAs, one commit: a
                // tcgen05 wait, fence or commit costs the issuing lane as much as several MMAs
                if (!wait_bar(bar + (kReady + s) * 8, (uint32_t)(u / kSB) & 1u, p, abt, 300 + u)) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                // B: K-major with the 128-byte swizzle: a token's 64 K in one 128-byte row, 1024
                // bytes between 8-token groups; step ks starts 32 bytes (16 K) into its half
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t baddr = b0 + (uint32_t)(s * C::kBStage + (ks >> 2) * C::kBHalf + (ks & 3) * 32);
                    const unsigned long long bdesc = (unsigned long long)((baddr & 0x3FFFFu) >> 4) |
                                                     (1ull << 16) | ((unsigned long long)(1024u >> 4) << 32) |
                                                     (1ull << 46) | (2ull << 61);
                    const uint32_t acc = (u > 0 || ks > 0) ? 1u : 0u;   // the first MMA overwrites
                    asm volatile("{\n .reg .pred pa;\n setp.ne.u32 pa, %4, 0;\n"
                                 " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, pa;\n}"
                                 ::"r"(tb), "r"(tb + C::kACol + 64u * (uint32_t)a + 8u * (uint32_t)ks),
                                   "l"(bdesc), "r"(C::kIdesc), "r"(acc) : "memory");
                }
                commit(bar + (kFree + s) * 8);   // the stage and the A slot (a == s)
                if (u == nst - 1) commit(bar + kDFull * 8);
            }
            // every MMA issued has completed before the tensor memory is released
            commit(bar + kDone * 8);
            wait_bar(bar + kDone * 8, 0u, p, nullptr, 500);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ dequantisation, then the epilogue
        const int q = warp & 3, blk = warp >> 2;        // lane quarter; block of the unit (32 K)
        const int r = 32 * q + lane;                    // this thread's row of the block
        const int tl = r >> 4, rit = r & 15;            // its tile of the block, row of the tile
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        bool ok = true;
        for (int u = 0; u < nst && ok; ++u) {
            const int s = u % kSW, a = u % kA;
            if (u >= kA && !warp_wait(bar + (kFree + a) * 8, (uint32_t)(u / kA - 1) & 1u, p, abt, 600 + u)) {
                ok = false;
                break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            if (!warp_wait(bar + (kWFull + s) * 8, (uint32_t)(u / kSW) & 1u, p, abt, 700 + u)) {
                ok = false;
                break;
            }
            const unsigned char* unit = smem + (size_t)s * kCodeBytes + (size_t)tl * kUnitBytes;
            const uint4 c4 = *reinterpret_cast<const uint4*>(unit + (blk * 16 + rit) * 16);
            const uint2 sc = *reinterpret_cast<const uint2*>(unit + 1024 + rit * 8);
            __syncwarp();
            if (lane == 0) arrive(bar + (kWEmpty + s) * 8);   // the codes are in registers
            const uint32_t sw = (blk & 2) ? sc.y : sc.x;
            const __half2 d2 = (blk & 1) ? __high2half2(as_h2(sw)) : __low2half2(as_h2(sw));
            const uint32_t ws[4] = {c4.x, c4.y, c4.z, c4.w};
            uint32_t v[16];
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                // byte j of a block holds codes j (low nibble) and j + 16 (high): the pairs
                // (4w, 4w + 1), (4w + 2, 4w + 3) and the same + 16, as columns 2w, 2w + 1,
                // 8 + 2w, 9 + 2w of the block
                const uint32_t r01 = __byte_perm(ws[w], 0u, 0x4140u), r23 = __byte_perm(ws[w], 0u, 0x4342u);
                v[2 * w] = deq2(r01, d2);
                v[2 * w + 1] = deq2(r23, d2);
                v[8 + 2 * w] = deq2(r01 >> 4, d2);
                v[9 + 2 * w] = deq2(r23 >> 4, d2);
            }
            asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
                         "%13,%14,%15,%16};"
                         ::"r"(tb + lane_base + C::kACol + 64u * (uint32_t)a + 16u * (uint32_t)blk), "r"(v[0]),
                           "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
                           "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]) : "memory");
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) arrive(bar + (kReady + a) * 8);
        }
        if (ok && warp_wait(bar + kDFull * 8, 0u, p, abt, 800)) {
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const int tile = rb * kRB + tl;
            const bool silu = p.silu != 0, split = p.kparts > 1;
            const int orow = silu ? tile * 8 + rit : tile * 16 + rit;   // output row
            const bool row_ok = split ? tile * 16 < p.R : silu ? (rit < 8 && orow < (p.rows >> 1)) : orow < p.rows;
            float* yf = static_cast<float*>(p.y);
            __half* yh = static_cast<__half*>(p.y);
            float* pf = split ? p.part + (size_t)kp * p.T * p.R + tile * 16 + rit : nullptr;
            // 32-column loads of the accumulator: NT / 128 per warp (NT = 32: the first warp of a
            // lane quarter takes the only one)
            constexpr int kLoads = NT / 32, kPerWarp = kLoads >= 4 ? kLoads / 4 : 1;
#pragma unroll 1
            for (int c = blk * kPerWarp; c < (blk + 1) * kPerWarp && c < kLoads; ++c) {
                uint32_t v[32];
                asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
                             "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                             : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
                               "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
                               "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
                               "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
                               "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
                             : "r"(tb + lane_base + 32u * (uint32_t)c) : "memory");
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int t = n0 + 32 * c + j;
                    const float val = __uint_as_float(v[j]);
                    const float up = __shfl_down_sync(0xffffffffu, val, 8);   // the up row of a gate row
                    if (!row_ok || t >= p.T) continue;
                    if (split) {   // the raw sum; the merge applies the epilogue
                        pf[(size_t)t * p.R] = val;
                        continue;
                    }
                    const size_t o = (size_t)t * p.ld + orow;
                    if (silu) yh[o] = __float2half_rn(persist::silu(val) * up);
                    else if (p.epi == QL_EPI_ADD_RESIDUAL) yf[o] = yf[o] + val;
                    else yf[o] = val;
                }
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tb), "r"(kTmemCols) : "memory");
    }
    // copies still in flight (only after an abort): the last use of each stage lands before the
    // CTA leaves (bounded)
    if (warp == kWProdWarp && lane == 0) {
        const int n = issued_w > prew ? issued_w : prew;
        for (int u = n - kSW < 0 ? 0 : n - kSW; u < n; ++u)
            wait_bar(bar + (kWFull + u % kSW) * 8, (uint32_t)(u / kSW) & 1u, p, nullptr, 900 + u);
    }
    if (warp == kBProdWarp && lane == 0) {
        const int n = issued_b;
        for (int u = n - kSB < 0 ? 0 : n - kSB; u < n; ++u)
            wait_bar(bar + (kReady + u % kSB) * 8, (uint32_t)(u / kSB) & 1u, p, nullptr, 1000 + u);
    }
}

// The K parts of a split GEMM added in part order (deterministic), then the epilogue. Grid
// (output rows / 1024, tokens): a thread takes 4 consecutive output rows of one token (4
// consecutive rows of the stream, SiLU*up: of a tile's gate rows, the up rows 8 further), and
// the loads of all its parts are in flight together.
constexpr int kMaxParts = 4;
__global__ void __launch_bounds__(256) gemm_merge_kernel(const __grid_constant__ Params p) {
    pdl_wait();
    pdl_trigger();
    const bool silu = p.silu != 0;
    const int orows = silu ? p.rows >> 1 : p.rows;
    const int t = blockIdx.y, j0 = (blockIdx.x * 256 + threadIdx.x) * 4;
    if (j0 >= orows) return;
    const int r0 = silu ? (j0 >> 3) * 16 + (j0 & 7) : j0;
    const float* q = p.part + (size_t)t * p.R + r0;
    const size_t ps = (size_t)p.T * p.R;
    float4 g[kMaxParts], u[kMaxParts];
#pragma unroll
    for (int k = 0; k < kMaxParts; ++k) {
        g[k] = u[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k < p.kparts) {
            g[k] = __ldcg(reinterpret_cast<const float4*>(q + k * ps));
            if (silu) u[k] = __ldcg(reinterpret_cast<const float4*>(q + k * ps + 8));
        }
    }
    float4 sg = g[0], su = u[0];
#pragma unroll
    for (int k = 1; k < kMaxParts; ++k) {
        if (k < p.kparts) {
            sg.x += g[k].x; sg.y += g[k].y; sg.z += g[k].z; sg.w += g[k].w;
            su.x += u[k].x; su.y += u[k].y; su.z += u[k].z; su.w += u[k].w;
        }
    }
    const float gv[4] = {sg.x, sg.y, sg.z, sg.w}, uv[4] = {su.x, su.y, su.z, su.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (j0 + i >= orows) break;
        const size_t o = (size_t)t * p.ld + j0 + i;
        if (silu) static_cast<__half*>(p.y)[o] = __float2half_rn(persist::silu(gv[i]) * uv[i]);
        else if (p.epi == QL_EPI_ADD_RESIDUAL) static_cast<float*>(p.y)[o] += gv[i];
        else static_cast<float*>(p.y)[o] = gv[i];
    }
}

}  // namespace gemm

namespace {

template <int NT>
cudaError_t gemm_attr(int optin) {
    cudaFuncAttributes fa = {};
    cudaError_t e = cudaFuncGetAttributes(&fa, gemm::gemm_tc_kernel<NT>);
    if (e == cudaSuccess && gemm::Cfg<NT>::kSmem + fa.sharedSizeBytes > (size_t)optin) e = cudaErrorInvalidConfiguration;
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm::gemm_tc_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)gemm::Cfg<NT>::kSmem);
    return e;
}

int gemm_prepare() {
    static std::mutex mu;
    static std::set<int> done;
    int dev = 0;
    QL_TRY_CUDA(cudaGetDevice(&dev));
    std::lock_guard<std::mutex> lk(mu);
    if (done.count(dev)) return QL_OK;
    int optin = 0;
    cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e == cudaSuccess) e = gemm_attr<32>(optin);
    if (e == cudaSuccess) e = gemm_attr<128>(optin);
    if (e == cudaSuccess) e = gemm_attr<256>(optin);
    if (e != cudaSuccess) return cuda_error(e, "gemm: kernel attributes");
    done.insert(dev);
    return QL_OK;
}

}  // namespace

int gemm_tc_launch(const GemmArgs& a, cudaStream_t s, bool pdl) {
    const PMat& M = a.M;
    QL_REQUIRE(M.stream != nullptr && M.nblk % 4 == 0 && M.nblk >= 4, "gemm: the tile stream copy, cols % 128 == 0");
    QL_REQUIRE(a.T >= 1 && a.x16 && a.y, "gemm: T >= 1 tokens, non-null input and output");
    QL_REQUIRE((reinterpret_cast<uintptr_t>(a.x16) & 15) == 0 && (reinterpret_cast<uintptr_t>(M.stream) & 15) == 0,
               "gemm: the activations and the stream must be 16-byte aligned");
    QL_REQUIRE(a.epi == QL_EPI_NONE || a.epi == QL_EPI_ADD_RESIDUAL || a.epi == QL_EPI_SILU_MUL, "gemm: unknown epilogue");
    QL_REQUIRE((a.epi == QL_EPI_SILU_MUL) == (M.silu != 0), "gemm: SiLU*up needs a matrix packed for it");
    DevError* err = device_error_record();
    if (!err) return set_error(QL_ECUDA, "gemm: no device error record");
    if (int rc = gemm_prepare()) return rc;
    gemm::Params p = {};
    if (int rc = q4_stream_tensor_map(M, &p.tw)) return rc;
    const uint64_t K = (uint64_t)M.nblk * 32;
    const int nt = a.T > 128 ? 256 : a.T > 32 ? 128 : 32;   // tokens per CTA: the weights read once per nt tokens
    if (int rc = f16_rows_tensor_map(a.x16, K, (uint64_t)a.T, 64, (uint32_t)nt, &p.tx, true)) return rc;
    p.T = a.T;
    p.rows = M.rows;
    p.nst = M.nblk / 4;
    p.silu = M.silu;
    p.epi = a.epi;
    p.ld = a.ld;
    p.y = a.y;
    p.err = err;
    p.timeout_ns = 2000000000ull;
    p.R = M.ntile * 16;
    // K parts: enough CTAs for the SMs when the matrix has few row blocks, at least 4 units each,
    // as many as the workspace holds
    const int nrb = (M.ntile + gemm::kRB - 1) / gemm::kRB, ntok = (a.T + nt - 1) / nt;
    int kparts = 1;
    if (a.part != nullptr) {
        kparts = num_sms() / (nrb * ntok);
        if (kparts > gemm::kMaxParts) kparts = gemm::kMaxParts;
        if (kparts > p.nst / 4) kparts = p.nst / 4;
        while (kparts > 1 && (size_t)kparts * a.T * p.R * sizeof(float) > a.part_bytes) --kparts;
        if (kparts < 1) kparts = 1;
    }
    p.upp = (p.nst + kparts - 1) / kparts;
    kparts = (p.nst + p.upp - 1) / p.upp;   // (no empty part)
    p.kparts = kparts;
    p.part = kparts > 1 ? a.part : nullptr;
    const dim3 grid((unsigned)nrb, (unsigned)ntok, (unsigned)kparts);
    cudaError_t e = nt == 256  ? ql::launch(gemm::gemm_tc_kernel<256>, grid, dim3(gemm::kThreads),
                                            gemm::Cfg<256>::kSmem, s, pdl, p)
                    : nt == 128 ? ql::launch(gemm::gemm_tc_kernel<128>, grid, dim3(gemm::kThreads),
                                             gemm::Cfg<128>::kSmem, s, pdl, p)
                                : ql::launch(gemm::gemm_tc_kernel<32>, grid, dim3(gemm::kThreads),
                                             gemm::Cfg<32>::kSmem, s, pdl, p);
    if (e != cudaSuccess) return cuda_error(e, "gemm launch");
    if (kparts > 1) {
        const int orows = M.silu ? M.rows / 2 : M.rows;
        e = ql::launch(gemm::gemm_merge_kernel, dim3((unsigned)((orows + 1023) / 1024), (unsigned)a.T), dim3(256), 0, s,
                       pdl, p);
        if (e != cudaSuccess) return cuda_error(e, "gemm merge launch");
    }
    return QL_OK;
}

}  // namespace ql

// ---------------------------------------------------------------------------------------------
// C ABI
extern "C" int ql_gemm_q4_0_stream(const void* d_stream, int64_t rows, int64_t cols, const void* d_x, int64_t n_tokens,
                                   void* d_y, int epilogue, void* stream) {
    using namespace ql;
    QL_REQUIRE(d_stream && d_x && d_y, "ql_gemm_q4_0_stream: null pointer");
    QL_REQUIRE(epilogue == QL_EPI_NONE || epilogue == QL_EPI_ADD_RESIDUAL || epilogue == QL_EPI_SILU_MUL,
               "ql_gemm_q4_0_stream: unknown epilogue");
    const int silu = epilogue == QL_EPI_SILU_MUL;
    QL_REQUIRE(rows > 0 && cols > 0 && cols % 128 == 0 && rows < (1ll << 30) && cols < (1ll << 24) && (!silu || rows % 2 == 0),
               "ql_gemm_q4_0_stream: need cols % 128 == 0 (and even rows with SiLU*up)");
    QL_REQUIRE(n_tokens >= 1 && n_tokens <= (1ll << 20), "ql_gemm_q4_0_stream: n_tokens must be in [1, 2^20]");
    QL_REQUIRE((reinterpret_cast<uintptr_t>(d_y) & 3) == 0, "ql_gemm_q4_0_stream: y must be 4-byte aligned");
    GemmArgs a = {};
    a.M.stream = static_cast<const uint8_t*>(d_stream);
    a.M.rows = (int)rows;
    a.M.nblk = (int)(cols / 32);
    a.M.silu = silu;
    a.M.ntile = silu ? (int)((rows / 2 + 7) / 8) : (int)((rows + 15) / 16);
    a.T = (int)n_tokens;
    a.x16 = static_cast<const __half*>(d_x);
    a.y = d_y;
    a.ld = (int)(silu ? rows / 2 : rows);
    a.epi = epilogue;
    return gemm_tc_launch(a, static_cast<cudaStream_t>(stream), true);
}
