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
// One CTA per (block of 128 weight rows = 8 tiles, tile of 128 tokens); K streams in units of
// 128 columns (one 1152-byte unit of each tile):
//  * warp 5, lane 0: per unit, one tensor-map copy of the row block's 8 tiles x 1 unit of codes
//    and scales (tiles past the matrix read as zero) and 16 tensor-map copies of the tokens'
//    activations (8 f16 of K x 128 tokens each: K-major core matrices, tokens past the chunk
//    read as zero) into a ring of kS stages, completing on the stage's mbarrier. The weight
//    copies of the first stages go out before the wait on the previous kernel;
//  * warps 0-3 (warp q serves tensor-memory lanes 32q..32q+31, i.e. rows 32q.. of the block):
//    each thread expands its row's 128 codes of the unit into (q - 8) d in f16, in K order
//    (two consecutive K per 32-bit column), and stores them into one of kA A slots of tensor
//    memory; after the last unit they run the epilogue;
//  * warp 4 allocates the tensor memory; its lane 0 issues tcgen05.mma (kind::f16, M 128, N 128,
//    K 16, A in tensor memory, B in shared memory) into one f32 accumulator of 128 columns and
//    commits each unit's MMAs to the barriers that free the unit's stage and A slot;
//  * epilogue: tcgen05.ld of the accumulator (a thread holds its row's 128 tokens), then the
//    stores: f32, added to the residual, or SiLU(gate) * up in f16 (the gate row's thread takes
//    the up row from the lane 8 above).
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
constexpr int kN = 128;                            // tokens per CTA: the MMA's N
constexpr int kS = 4;                              // ring stages
constexpr int kA = 4;                              // A slots of tensor memory, one unit (64 columns) each
constexpr int kCodeBytes = kRB * kUnitBytes;       // 9216
constexpr int kChunkBytes = kN * 16;               // 8 f16 of K for 128 tokens
constexpr int kBBytes = 16 * kChunkBytes;          // the unit's 128 K for 128 tokens
constexpr int kStage = kCodeBytes + kBBytes;       // a multiple of 128
constexpr size_t kSmem = (size_t)kS * kStage;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kACol = kN;                     // the A slots after the accumulator's columns
// instruction descriptor: D f32, A and B f16, both K-major, N = 128, M = 128
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(kN >> 3) << 17) | ((128u >> 4) << 24);
constexpr int kMmaWarp = 4, kProdWarp = 5, kThreads = 6 * 32;
enum { kFull = 0, kEmpty = kS, kAFull = 2 * kS, kAFree = 2 * kS + kA, kDFull = 2 * kS + 2 * kA, kDone = kDFull + 1,
       kBars = kDone + 1 };
static_assert(kStage % 128 == 0 && kCodeBytes % 128 == 0, "stage regions 128-byte aligned");
static_assert(kACol + kA * 64 <= kTmemCols, "tensor memory: accumulator + A slots");

struct Params {
    CUtensorMap tw;       // weights: [tile][unit][144 x 8 B], boxes of 8 tiles x 1 unit
    CUtensorMap tx;       // activations: [T][K] f16, boxes of 128 tokens x 8
    int T, rows, nst, silu, epi, ld;
    void* y;
    DevError* err;
    unsigned long long timeout_ns;
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

// wait_bar by every lane, one answer for the warp (its collective tcgen05 instructions need
// every lane or none)
__device__ __forceinline__ bool warp_wait(uint32_t mb, uint32_t parity, const Params& p, int* abort_flag, int where) {
    const bool ok = wait_bar(mb, parity, p, abort_flag, where);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void arrive(uint32_t mb) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mb) : "memory");
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

__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ __align__(8) unsigned long long bars[kBars];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ int issued_units;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rb = blockIdx.x, n0 = blockIdx.y * kN, nst = p.nst;
    const uint32_t bar = su32(bars);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kS; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar + (kFull + s) * 8) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar + (kEmpty + s) * 8) : "memory");
        }
        for (int a = 0; a < kA; ++a) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;" ::"r"(bar + (kAFull + a) * 8) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar + (kAFree + a) * 8) : "memory");
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar + kDFull * 8) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar + kDone * 8) : "memory");
        abort_flag = 0;
        issued_units = 0;
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

    // the weight copy of unit u into stage u % kS, and the activation copies (16 chunks of 8 K)
    auto copy_w = [&](int u, unsigned long long pol) {
        const int s = u % kS;
        asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
                     " [%0], [%1, {%2, %3, %4}], [%5], %6;"
                     ::"r"(su32(smem + (size_t)s * kStage)), "l"(reinterpret_cast<uint64_t>(&p.tw)), "r"(0), "r"(u),
                       "r"(rb * kRB), "r"(bar + (kFull + s) * 8), "l"(pol) : "memory");
    };
    auto copy_x = [&](int u) {
        const int s = u % kS;
        const uint32_t dst = su32(smem + (size_t)s * kStage + kCodeBytes);
        for (int c = 0; c < 16; ++c)
            asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                         " [%0], [%1, {%2, %3}], [%4];"
                         ::"r"(dst + (uint32_t)(c * kChunkBytes)), "l"(reinterpret_cast<uint64_t>(&p.tx)),
                           "r"(128 * u + 8 * c), "r"(n0), "r"(bar + (kFull + s) * 8) : "memory");
    };
    const int pre = nst < kS ? nst : kS;
    unsigned long long pol = 0;
    if (warp == kProdWarp && lane == 0) {
        pol = l2_evict_first();
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tw)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tx)) : "memory");
        // the weights do not depend on the previous kernel: the first stages' codes go out now
        for (int u = 0; u < pre; ++u) {
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar + (kFull + u) * 8),
                         "r"((uint32_t)kStage) : "memory");
            copy_w(u, pol);
        }
    }
    pdl_wait();
    pdl_trigger();

    if (warp == kProdWarp) {
        // ------------------------------------------------ copies (one lane)
        if (lane == 0) {
            int u = 0;
            for (; u < pre; ++u) copy_x(u);
            for (; u < nst; ++u) {
                const int s = u % kS;
                if (!wait_bar(bar + (kEmpty + s) * 8, (uint32_t)(u / kS - 1) & 1u, p, abt, 100 + u)) break;
                // the stage's codes were read through the generic proxy; the copies write it
                // through the async proxy
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar + (kFull + s) * 8),
                             "r"((uint32_t)kStage) : "memory");
                copy_w(u, pol);
                copy_x(u);
            }
            issued_units = u;
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------ MMA issue (one lane)
        if (lane == 0) {
            const uint32_t sb = su32(smem);
            for (int u = 0; u < nst; ++u) {
                const int s = u % kS, a = u % kA;
                if (!wait_bar(bar + (kAFull + a) * 8, (uint32_t)(u / kA) & 1u, p, abt, 200 + u)) break;
                if (!wait_bar(bar + (kFull + s) * 8, (uint32_t)(u / kS) & 1u, p, abt, 300 + u)) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                // B: K-major core matrices, 2048 bytes between the K halves of a step (a chunk of 8
                // K for 128 tokens), 128 bytes between 8-token groups; step ks starts 2 chunks in
                const uint32_t b0 = sb + (uint32_t)(s * kStage + kCodeBytes);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t baddr = b0 + (uint32_t)(ks * 2 * kChunkBytes);
                    const unsigned long long bdesc = (unsigned long long)((baddr & 0x3FFFFu) >> 4) |
                                                     ((unsigned long long)(kChunkBytes >> 4) << 16) |
                                                     ((unsigned long long)(128u >> 4) << 32) | (1ull << 46);
                    const uint32_t acc = (u > 0 || ks > 0) ? 1u : 0u;   // the first MMA overwrites
                    asm volatile("{\n .reg .pred pa;\n setp.ne.u32 pa, %4, 0;\n"
                                 " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, pa;\n}"
                                 ::"r"(tb), "r"(tb + kACol + 64u * (uint32_t)a + 8u * (uint32_t)ks), "l"(bdesc),
                                   "r"(kIdesc), "r"(acc) : "memory");
                }
                commit(bar + (kEmpty + s) * 8);   // the stage (codes already read, activations read now)
                commit(bar + (kAFree + a) * 8);
                if (u == nst - 1) commit(bar + kDFull * 8);
            }
            // every MMA issued has completed before the tensor memory is released
            commit(bar + kDone * 8);
            wait_bar(bar + kDone * 8, 0u, p, nullptr, 400);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ dequantisation, then the epilogue
        const int q = warp, r = 32 * q + lane;          // this thread's row of the block
        const int tl = r >> 4, rit = r & 15;            // its tile of the block, row of the tile
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        bool ok = true;
        for (int u = 0; u < nst && ok; ++u) {
            const int s = u % kS, a = u % kA;
            if (u >= kA && !warp_wait(bar + (kAFree + a) * 8, (uint32_t)(u / kA - 1) & 1u, p, abt, 500 + u)) {
                ok = false;
                break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            if (!warp_wait(bar + (kFull + s) * 8, (uint32_t)(u / kS) & 1u, p, abt, 600 + u)) {
                ok = false;
                break;
            }
            const unsigned char* unit = smem + (size_t)s * kStage + (size_t)tl * kUnitBytes;
            uint4 cw[4];
#pragma unroll
            for (int b = 0; b < 4; ++b) cw[b] = *reinterpret_cast<const uint4*>(unit + (b * 16 + rit) * 16);
            const uint2 sc = *reinterpret_cast<const uint2*>(unit + 1024 + rit * 8);
#pragma unroll
            for (int half = 0; half < 2; ++half) {   // blocks 2 half, 2 half + 1: 64 K, 32 columns
                uint32_t v[32];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const uint4 c4 = cw[2 * half + e];
                    const uint32_t sw = half ? sc.y : sc.x;
                    const __half2 d2 = e ? __high2half2(as_h2(sw)) : __low2half2(as_h2(sw));
                    const uint32_t ws[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        // byte j of a block holds codes j (low nibble) and j + 16 (high): the pairs
                        // (4w, 4w + 1), (4w + 2, 4w + 3) and the same + 16, as columns 2w, 2w + 1,
                        // 8 + 2w, 9 + 2w of the block
                        const uint32_t r01 = __byte_perm(ws[w], 0u, 0x4140u), r23 = __byte_perm(ws[w], 0u, 0x4342u);
                        v[16 * e + 2 * w] = deq2(r01, d2);
                        v[16 * e + 2 * w + 1] = deq2(r23, d2);
                        v[16 * e + 8 + 2 * w] = deq2(r01 >> 4, d2);
                        v[16 * e + 9 + 2 * w] = deq2(r23 >> 4, d2);
                    }
                }
                asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
                             "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
                             ::"r"(tb + lane_base + kACol + 64u * (uint32_t)a + 32u * (uint32_t)half), "r"(v[0]),
                               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
                               "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
                               "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]),
                               "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]),
                               "r"(v[30]), "r"(v[31]) : "memory");
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) arrive(bar + (kAFull + a) * 8);
        }
        if (ok && warp_wait(bar + kDFull * 8, 0u, p, abt, 700)) {
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const int tile = rb * kRB + tl;
            const bool silu = p.silu != 0;
            const int orow = silu ? tile * 8 + rit : tile * 16 + rit;   // output row
            const bool row_ok = silu ? (rit < 8 && orow < (p.rows >> 1)) : orow < p.rows;
            float* yf = static_cast<float*>(p.y);
            __half* yh = static_cast<__half*>(p.y);
#pragma unroll 1
            for (int c = 0; c < kN / 32; ++c) {   // 32 tokens at a time
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
    if (warp == kProdWarp && lane == 0) {
        const int n = issued_units > pre ? issued_units : pre;
        for (int u = n - kS < 0 ? 0 : n - kS; u < n; ++u)
            wait_bar(bar + (kFull + u % kS) * 8, (uint32_t)(u / kS) & 1u, p, nullptr, 800 + u);
    }
}

}  // namespace gemm

namespace {

int gemm_prepare() {
    static std::mutex mu;
    static std::set<int> done;
    int dev = 0;
    QL_TRY_CUDA(cudaGetDevice(&dev));
    std::lock_guard<std::mutex> lk(mu);
    if (done.count(dev)) return QL_OK;
    int optin = 0;
    cudaFuncAttributes fa = {};
    cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, gemm::gemm_tc_kernel);
    if (e == cudaSuccess && gemm::kSmem + fa.sharedSizeBytes > (size_t)optin) e = cudaErrorInvalidConfiguration;
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemm::gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gemm::kSmem);
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
    if (int rc = f16_rows_tensor_map(a.x16, K, (uint64_t)a.T, 8, gemm::kN, &p.tx)) return rc;
    p.T = a.T;
    p.rows = M.rows;
    p.nst = M.nblk / 4;
    p.silu = M.silu;
    p.epi = a.epi;
    p.ld = a.ld;
    p.y = a.y;
    p.err = err;
    p.timeout_ns = 2000000000ull;
    const dim3 grid((unsigned)((M.ntile + gemm::kRB - 1) / gemm::kRB), (unsigned)((a.T + gemm::kN - 1) / gemm::kN));
    const cudaError_t e = ql::launch(gemm::gemm_tc_kernel, grid, dim3(gemm::kThreads), gemm::kSmem, s, pdl, p);
    return e == cudaSuccess ? QL_OK : cuda_error(e, "gemm launch");
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
