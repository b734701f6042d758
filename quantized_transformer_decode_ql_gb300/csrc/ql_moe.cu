// Routed experts (MoE) of a Qwen3-MoE-style layer at batch 1: the router with its top-k, and the
// weighted combination of the selected experts' outputs into the residual stream. The experts'
// own GEMVs are the stream GEMV over a selection of experts (ql_persist.cuh, PMat::sel).
//
// [IL] inferencelayer cuda_llm.rs: Cfg (num_experts, topk, moe_inter, norm_topk; no shared
// expert) and the MoE branch of CudaQwen3::step: router logits from the f32 router weights and
// the normalised input, a top-k with weights, gate|up and down over the selected experts,
// then a combine into the residual. The page does not print its topk kernel; the reading
// taken: the softmax over all experts' logits, the k largest (the lowest index first among
// equal values), their probabilities renormalised to sum 1 when norm_topk is set.
#include <cuda_fp16.h>
#include <math.h>

#include <cstdlib>

#include "ql_internal.h"

namespace ql {
namespace {

constexpr int kRouterWarps = 8;
constexpr int kMaxExpertsPerLane = 16;   // E <= 512

// One warp per expert row: logit[e] = rs * sum_i (router[e][i] w[i]) x[i] (the RMSNorm'd input,
// rs from the CTA's own sum of squares). CH > 0: the row times the norm weight (both constants of
// the step) is loaded into registers before the wait on the predecessor, CH float4 per lane
// (hidden = 128 CH); CH = 0 loads it after the wait. The CTA that takes the last ticket selects
// the top-k.
template <int CH>
__global__ void __launch_bounds__(kRouterWarps * 32) moe_router_kernel(MoeRouterArgs a, DevError* err) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int e = blockIdx.x * kRouterWarps + warp;
    float4 rw[CH > 0 ? CH : 1];
    if (CH > 0 && e < a.num_experts) {
        const float* r = a.router + (size_t)e * a.hidden;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const float4 rv = __ldg(reinterpret_cast<const float4*>(r + lane * 4 + 128 * c));
            const float4 wv = __ldg(reinterpret_cast<const float4*>(a.norm_w + lane * 4 + 128 * c));
            rw[c] = make_float4(rv.x * wv.x, rv.y * wv.y, rv.z * wv.z, rv.w * wv.w);
        }
    }
    pdl_wait();
    pdl_trigger();
    __shared__ float red[kRouterWarps];
    __shared__ int last;
    // the RMSNorm scale of x (every CTA computes it; x is 4 * hidden bytes in L2)
    float ss = 0.f;
    for (int i = tid * 4; i < a.hidden; i += kRouterWarps * 32 * 4) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(a.x + i));
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kRouterWarps; ++w) tot += red[w];
    const float rs = rsqrtf(fmaf(tot, 1.0f / (float)a.hidden, a.eps));
    if (e < a.num_experts) {
        float dot = 0.f;
        if (CH > 0) {
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                const float4 xv = __ldcg(reinterpret_cast<const float4*>(a.x + lane * 4 + 128 * c));
                dot = fmaf(rw[c].x, xv.x, dot);
                dot = fmaf(rw[c].y, xv.y, dot);
                dot = fmaf(rw[c].z, xv.z, dot);
                dot = fmaf(rw[c].w, xv.w, dot);
            }
        } else {
            const float* r = a.router + (size_t)e * a.hidden;
            for (int i = lane * 4; i < a.hidden; i += 128) {
                const float4 rv = __ldg(reinterpret_cast<const float4*>(r + i));
                const float4 xv = __ldcg(reinterpret_cast<const float4*>(a.x + i));
                const float4 wv = __ldg(reinterpret_cast<const float4*>(a.norm_w + i));
                dot = fmaf(rv.x * wv.x, xv.x, dot);
                dot = fmaf(rv.y * wv.y, xv.y, dot);
                dot = fmaf(rv.z * wv.z, xv.z, dot);
                dot = fmaf(rv.w * wv.w, xv.w, dot);
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        if (lane == 0) a.logits[e] = dot * rs;
    }
    // the last CTA (an acq_rel ticket orders every CTA's logits before its reads) selects
    __syncthreads();
    if (tid == 0) {
        int t;
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(t) : "l"(a.ticket) : "memory");
        last = t == (int)gridDim.x - 1;
    }
    __syncthreads();
    if (!last || warp != 0) return;
    const int E = a.num_experts;
    float l[kMaxExpertsPerLane];
    float m = -INFINITY;
#pragma unroll
    for (int c = 0; c < kMaxExpertsPerLane; ++c) {
        const int i = lane + 32 * c;
        l[c] = i < E ? __ldcg(a.logits + i) : -INFINITY;
        m = fmaxf(m, l[c]);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float sum = 0.f;
#pragma unroll
    for (int c = 0; c < kMaxExpertsPerLane; ++c) sum += lane + 32 * c < E ? expf(l[c] - m) : 0.f;
#pragma unroll
    for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    // k rounds of a warp argmax (the larger logit, else the lower index), the winner removed
    float wsum = 0.f;
    for (int j = 0; j < a.topk; ++j) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int c = 0; c < kMaxExpertsPerLane; ++c) {
            const int i = lane + 32 * c;
            if (i < E && (l[c] > bv || (l[c] == bv && i < bi))) {
                bv = l[c];
                bi = i;
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if (bi < 0 || bi >= E) {   // fewer experts than k (validated on the host): keep in range
            if (lane == 0) record_device_error(err, kErrMoeExpert, j, bi);
            bi = 0;
        }
#pragma unroll
        for (int c = 0; c < kMaxExpertsPerLane; ++c)
            if (lane + 32 * c == bi) l[c] = -INFINITY;
        const float p = expf(bv - m) / sum;
        wsum += p;
        if (lane == 0) {
            a.eidx[j] = bi;
            a.ewt[j] = p;
        }
    }
    __syncwarp();
    if (a.norm_topk && lane == 0) {
        const float inv = 1.0f / wsum;
        for (int j = 0; j < a.topk; ++j) a.ewt[j] *= inv;
    }
    if (lane == 0) *a.ticket = 0;   // re-armed for the next layer / step
}

// The cluster form (at most 128 experts, top-k at most 32, hidden = 128 CH): the router's CTAs,
// 16 warps each, one warp per expert, are one thread-block cluster of at most 8. A warp loads its
// expert's router row times the norm weight before the wait, then all of x once after it: the
// sum of squares (the RMSNorm scale; every warp holds the whole vector) and the dot product come
// from the same loads, with no CTA-wide step. The logits stay in shared memory; after a cluster
// barrier warp 0 of the CTA of rank 0 reads all of them through distributed shared memory
// (`mapa`, `ld.shared::cluster`) and selects the top-k with warp reductions (redux.sync) on
// order-preserving integer keys of the logits; a second barrier keeps every CTA's logits alive
// until they are read. No global round trip between the logits and the selection.
constexpr int kRouterClWarps = 16, kRouterClMaxCtas = 8;
__device__ __forceinline__ void cl_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cl_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// order-preserving key of a float (larger float, larger key); NaN below everything
__device__ __forceinline__ unsigned int logit_key(float f) {
    if (f != f) return 0u;
    const unsigned int u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_logit(unsigned int k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

template <int CH>
__global__ void __launch_bounds__(kRouterClWarps * 32) moe_router_cluster_kernel(MoeRouterArgs a, DevError* err) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int e = blockIdx.x * kRouterClWarps + warp;
    const bool own = e < a.num_experts;
    __shared__ float lg[kRouterClWarps];
    float4 rw[CH];
    if (own) {
        const float* r = a.router + (size_t)e * a.hidden;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const float4 rv = __ldg(reinterpret_cast<const float4*>(r + lane * 4 + 128 * c));
            const float4 wv = __ldg(reinterpret_cast<const float4*>(a.norm_w + lane * 4 + 128 * c));
            rw[c] = make_float4(rv.x * wv.x, rv.y * wv.y, rv.z * wv.z, rv.w * wv.w);
        }
    }
    pdl_wait();
    pdl_trigger();
    if (own) {
        float ss = 0.f, dot = 0.f;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const float4 xv = __ldcg(reinterpret_cast<const float4*>(a.x + lane * 4 + 128 * c));
            ss += xv.x * xv.x + xv.y * xv.y + xv.z * xv.z + xv.w * xv.w;
            dot = fmaf(rw[c].x, xv.x, dot);
            dot = fmaf(rw[c].y, xv.y, dot);
            dot = fmaf(rw[c].z, xv.z, dot);
            dot = fmaf(rw[c].w, xv.w, dot);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            ss += __shfl_xor_sync(0xffffffffu, ss, o);
            dot += __shfl_xor_sync(0xffffffffu, dot, o);
        }
        if (lane == 0) lg[warp] = dot * rsqrtf(fmaf(ss, 1.0f / (float)a.hidden, a.eps));
    }
    cl_arrive();   // every CTA's logits are in its shared memory
    cl_wait();
    unsigned int rank;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    const bool selector = rank == 0 && warp == 0;
    const int E = a.num_experts;
    float l[4];   // expert lane + 32 c
    if (selector) {
        const uint32_t lg_s = static_cast<uint32_t>(__cvta_generic_to_shared(lg));
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int i = lane + 32 * c;
            float v = -INFINITY;
            if (i < E) {
                uint32_t addr;
                asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(addr)
                             : "r"(lg_s + (uint32_t)(i % kRouterClWarps) * 4u), "r"((uint32_t)(i / kRouterClWarps)));
                asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
            }
            l[c] = v;
        }
    }
    cl_arrive();   // the logits have been read: the other CTAs may leave
    if (selector) {
        float m = fmaxf(fmaxf(l[0], l[1]), fmaxf(l[2], l[3]));
#pragma unroll
        for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float sum = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) sum += lane + 32 * c < E ? expf(l[c] - m) : 0.f;
#pragma unroll
        for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        unsigned int key[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) key[c] = lane + 32 * c < E ? logit_key(l[c]) : 0u;
        // k rounds: the largest key, the lowest index among equal keys; the winner removed
        float wsum = 0.f, myp = 0.f;
        for (int j = 0; j < a.topk; ++j) {
            unsigned int bk = 0u, bi = 0xFFFFFFFFu;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const unsigned int i = (unsigned int)(lane + 32 * c);
                if ((int)i < E && (key[c] > bk || bi == 0xFFFFFFFFu)) {
                    bk = key[c];
                    bi = i;
                }
            }
            const unsigned int wk = __reduce_max_sync(0xffffffffu, bk);
            unsigned int wi = __reduce_min_sync(0xffffffffu, bk == wk ? bi : 0xFFFFFFFFu);
            if (wi >= (unsigned int)E) {   // fewer experts than k (validated on the host): keep in range
                if (lane == 0) record_device_error(err, kErrMoeExpert, j, (long long)wi);
                wi = 0u;
            }
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if ((unsigned int)(lane + 32 * c) == wi) key[c] = 0u;
            const float p = expf(key_logit(wk) - m) / sum;
            wsum += p;
            if (lane == j) myp = p;
            if (lane == 0) a.eidx[j] = (int32_t)wi;
        }
        if (lane < a.topk) a.ewt[lane] = a.norm_topk ? myp * (1.0f / wsum) : myp;
    }
    cl_wait();
}

// x[i] += sum_j ewt[j] * y[j][i], the selected experts in slot order.
__global__ void __launch_bounds__(256) moe_combine_kernel(float* x, const float* y, const float* ewt, int hidden,
                                                          int k) {
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= hidden) return;
    float acc = 0.f;
    for (int j = 0; j < k; ++j) acc = fmaf(__ldcg(ewt + j), __ldcg(y + (size_t)j * hidden + i), acc);
    x[i] += acc;
}

}  // namespace

int moe_router_launch(const MoeRouterArgs& a, cudaStream_t s, bool pdl) {
    QL_REQUIRE(a.x && a.norm_w && a.router && a.logits && a.ticket && a.eidx && a.ewt, "moe router: null pointer");
    QL_REQUIRE(a.num_experts >= 1 && a.num_experts <= 32 * kMaxExpertsPerLane, "moe router: 1..512 experts");
    QL_REQUIRE(a.topk >= 1 && a.topk <= a.num_experts && a.topk <= 64, "moe router: bad top-k");
    QL_REQUIRE(a.hidden % 128 == 0, "moe router: hidden must be a multiple of 128");
    DevError* err = device_error_record();
    if (!err) return set_error(QL_ECUDA, "moe router: no device error record");
    const int ch = a.hidden / 128;
    // the cluster form: the CTAs of the router as one cluster, the selection through distributed
    // shared memory (QL_MOE_ROUTER_TICKET=1 keeps the ticket form for A/B measurements)
    static const bool ticket_only = [] {
        const char* e = std::getenv("QL_MOE_ROUTER_TICKET");
        return e && std::atoi(e) != 0;
    }();
    const int cl_ctas = (a.num_experts + kRouterClWarps - 1) / kRouterClWarps;
    if (!ticket_only && cl_ctas <= kRouterClMaxCtas && a.topk <= 32 && (ch == 16 || ch == 8 || ch == 2)) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cl_ctas);
        cfg.blockDim = dim3(kRouterClWarps * 32);
        cfg.stream = s;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cl_ctas;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 2 : 1;
        const cudaError_t e = ch == 16  ? cudaLaunchKernelEx(&cfg, moe_router_cluster_kernel<16>, a, err)
                              : ch == 8 ? cudaLaunchKernelEx(&cfg, moe_router_cluster_kernel<8>, a, err)
                                        : cudaLaunchKernelEx(&cfg, moe_router_cluster_kernel<2>, a, err);
        return e == cudaSuccess ? QL_OK : cuda_error(e, "moe router launch");
    }
    const int grid = (a.num_experts + kRouterWarps - 1) / kRouterWarps;
    const dim3 g(grid), b(kRouterWarps * 32);
    const cudaError_t e = ch == 16  ? launch(moe_router_kernel<16>, g, b, 0, s, pdl, a, err)
                          : ch == 8 ? launch(moe_router_kernel<8>, g, b, 0, s, pdl, a, err)
                          : ch == 2 ? launch(moe_router_kernel<2>, g, b, 0, s, pdl, a, err)
                                    : launch(moe_router_kernel<0>, g, b, 0, s, pdl, a, err);
    return e == cudaSuccess ? QL_OK : cuda_error(e, "moe router launch");
}

int moe_combine_launch(float* x, const float* y, const float* ewt, int hidden, int k, cudaStream_t s, bool pdl) {
    const cudaError_t e =
        launch(moe_combine_kernel, dim3((hidden + 255) / 256), dim3(256), 0, s, pdl, x, y, ewt, hidden, k);
    return e == cudaSuccess ? QL_OK : cuda_error(e, "moe combine launch");
}

}  // namespace ql
