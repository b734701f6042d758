// Paged split-K GQA decode attention over an f16 block pool.
//
// [FK] ferrum-kernels cuda_decode.rs: launch_paged_decode_attention / attention_paged (16-token
// blocks, block table, valid length = current length + 1, scale 1/sqrt(hd)) and the split-K
// flash-decode phase 1 + reduce; [IL] inferencelayer cuda_llm.rs CudaQwen3::step
// (attn_partial + attn_reduce over per-(head, chunk) running max / sum / weighted V).
//
// out[b][h] = sum_t softmax_t(q[b][h] . k[g][t] * scale) v[g][t], g = h / (n_heads / n_kv).
//
// Design (GB300): one CTA per (split, kv head, sequence), 4 warps. The CTA handles the whole
// GQA group of its kv head, so each K/V byte is read from HBM once and used by all G query
// heads. A warp takes one 16-token block at a time:
//  * scores: lane (t, half) = (lane & 15, lane >> 4) dots key t's half of head_dim against the
//    G queries (staged once in shared memory as f32), halves combined with one shuffle;
//  * online softmax per head in the exp2 domain (scores pre-scaled by scale * log2 e);
//  * P.V: lane owns head_dim/32 output dims of every head; probabilities go through a tiny
//    per-warp shared buffer (one broadcast load per key); V rows are read with coalesced
//    8-byte loads (256 contiguous bytes per key per warp at head_dim 128).
// The 4 warps' states are merged in shared memory; with one split the CTA writes the output,
// otherwise it writes its (m, l, acc) partial and the last CTA of its (sequence, kv head) -
// found with an atomic ticket, no waiting - merges all partials and re-arms the ticket.
#include <cuda_fp16.h>
#include <math.h>

#include "ql_internal.h"

namespace ql {
namespace {

constexpr int kAttnWarps = 4;
constexpr int kAttnThreads = kAttnWarps * 32;
constexpr int kBS = 16;   // tokens per KV block
constexpr int kMaxSplit = 256;   // splits per (sequence, kv head), bounded by the host

struct AParams {
    const __half* q;
    const __half* k_pool;
    const __half* v_pool;
    const int32_t* block_tables;
    const int32_t* context_lens;
    const int32_t* positions;
    const int32_t* active;
    int n_heads, n_kv, maxb;
    long long num_blocks;
    float scale_log2;   // scale * log2(e)
    __half* out;
    int* tickets;       // [batch][n_kv]
    float* pm;          // [batch][n_heads][nsplit]
    float* pl;
    float* pacc;        // [batch][n_heads][nsplit][HD]
    int nsplit, spb;
    int prefetch;       // warm L2 with this CTA's K/V tiles before waiting on the predecessor
};

__device__ __forceinline__ float2 h2f(uint32_t u) {
    __half2 h;
    *reinterpret_cast<uint32_t*>(&h) = u;
    return __half22float2(h);
}

template <int HD, int G>
__global__ void __launch_bounds__(kAttnThreads) attn_split_kernel(AParams p, DevError* err) {
    constexpr int HALF = HD / 2;         // dims per lane in the score phase
    constexpr int DPL = HD / 32;         // output dims per lane in the P.V phase
    __shared__ float q_s[G][HD];
    __shared__ float p_s[kAttnWarps][kBS][G];
    __shared__ float wm[kAttnWarps][G], wl[kAttnWarps][G];
    __shared__ float wacc[kAttnWarps][G][HD];
    __shared__ int last_flag;

    const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (p.prefetch && (p.active == nullptr || p.active[b] != 0)) {
        // In the decode step the context length comes from the position, which is final before
        // this kernel starts; only the newest slot is still being written (prefetch is a hint).
        const int Lp = p.positions[b] + 1;
        const int b0 = s * p.spb, b1 = min((Lp + kBS - 1) / kBS, b0 + p.spb);
        if (Lp <= p.maxb * kBS && (int)threadIdx.x < 2 * (b1 - b0) && b0 < b1) {
            const int blk = b0 + (threadIdx.x >> 1);
            const int phys = p.block_tables[(size_t)b * p.maxb + blk];
            if (phys >= 0 && phys < p.num_blocks) {
                const __half* base = (threadIdx.x & 1) ? p.v_pool : p.k_pool;
                const __half* t = base + ((size_t)phys * p.n_kv + g) * kBS * HD;
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(t), "r"((uint32_t)(kBS * HD * 2)) : "memory");
            }
        }
    }
    pdl_wait();
    pdl_trigger();
    if (p.active && p.active[b] == 0) return;
    const int L = p.context_lens ? p.context_lens[b] : p.positions[b] + 1;
    if (L <= 0) return;   // idle slot
    if (L > p.maxb * kBS) {
        if (s == 0 && threadIdx.x == 0) record_device_error(err, kErrAttnLength, b, L);
        return;
    }
    const int nblocks = (L + kBS - 1) / kBS;
    const int n_active = (nblocks + p.spb - 1) / p.spb;
    if (s >= n_active) return;
    const int blk0 = s * p.spb;
    const int blk1 = min(nblocks, blk0 + p.spb);

    for (int i = threadIdx.x; i < G * HD; i += kAttnThreads) {
        const int h = i / HD, d = i - h * HD;
        q_s[h][d] = __half2float(p.q[((size_t)b * p.n_heads + g * G + h) * HD + d]);
    }
    __syncthreads();

    float m[G], l[G], acc[G][DPL];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[h][e] = 0.f;
    }
    const int t = lane & 15, half = lane >> 4;
    const int32_t* bt = p.block_tables + (size_t)b * p.maxb;

    for (int blk = blk0 + warp; blk < blk1; blk += kAttnWarps) {
        const int phys = bt[blk];
        if (phys < 0 || phys >= p.num_blocks) {
            if (lane == 0) record_device_error(err, kErrAttnBlock, (long long)b * p.maxb + blk, phys);
            continue;
        }
        const size_t tile = ((size_t)phys * p.n_kv + g) * kBS * HD;
        const int nt = min(kBS, L - blk * kBS);      // valid keys in this block
        // ---- scores
        const uint4* kr = reinterpret_cast<const uint4*>(p.k_pool + tile + (size_t)t * HD + half * HALF);
        uint4 kv[HALF / 8];
#pragma unroll
        for (int c = 0; c < HALF / 8; ++c) kv[c] = kr[c];
        // V rows for this lane's output dims, all 16 keys (issued early)
        uint32_t vv[kBS][DPL / 2];
        const __half* vb = p.v_pool + tile + lane * DPL;
#pragma unroll
        for (int k = 0; k < kBS; ++k) {
            if (DPL == 4) {
                const uint2 u = *reinterpret_cast<const uint2*>(vb + (size_t)k * HD);
                vv[k][0] = u.x;
                if (DPL / 2 > 1) vv[k][DPL / 2 - 1] = u.y;
            } else {
                vv[k][0] = *reinterpret_cast<const uint32_t*>(vb + (size_t)k * HD);
            }
        }
        float sc[G];
#pragma unroll
        for (int h = 0; h < G; ++h) sc[h] = 0.f;
#pragma unroll
        for (int c = 0; c < HALF / 8; ++c) {
            const float2 k0 = h2f(kv[c].x), k1 = h2f(kv[c].y), k2 = h2f(kv[c].z), k3 = h2f(kv[c].w);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float* qq = &q_s[h][half * HALF + c * 8];
                float a = sc[h];
                a = fmaf(qq[0], k0.x, a); a = fmaf(qq[1], k0.y, a);
                a = fmaf(qq[2], k1.x, a); a = fmaf(qq[3], k1.y, a);
                a = fmaf(qq[4], k2.x, a); a = fmaf(qq[5], k2.y, a);
                a = fmaf(qq[6], k3.x, a); a = fmaf(qq[7], k3.y, a);
                sc[h] = a;
            }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
            sc[h] += __shfl_xor_sync(0xffffffffu, sc[h], 16);
            sc[h] = (t < nt) ? sc[h] * p.scale_log2 : -INFINITY;
        }
        // ---- online softmax (16 keys live in lanes 0..15, mirrored in 16..31)
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float mb = sc[h];
#pragma unroll
            for (int o = 8; o; o >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
            const float mn = fmaxf(m[h], mb);
            const float pr = exp2f(sc[h] - mn);
            float ls = pr;
#pragma unroll
            for (int o = 8; o; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
            const float alpha = exp2f(m[h] - mn);
            l[h] = l[h] * alpha + ls;
            m[h] = mn;
#pragma unroll
            for (int e = 0; e < DPL; ++e) acc[h][e] *= alpha;
            if (half == 0) p_s[warp][t][h] = pr;
        }
        __syncwarp();
        // ---- P.V
#pragma unroll
        for (int k = 0; k < kBS; ++k) {
            if (k < nt) {
                float pv[G];
#pragma unroll
                for (int h = 0; h < G; ++h) pv[h] = p_s[warp][k][h];
#pragma unroll
                for (int e2 = 0; e2 < DPL / 2; ++e2) {
                    const float2 v = h2f(vv[k][e2]);
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        acc[h][2 * e2] = fmaf(pv[h], v.x, acc[h][2 * e2]);
                        acc[h][2 * e2 + 1] = fmaf(pv[h], v.y, acc[h][2 * e2 + 1]);
                    }
                }
            }
        }
        __syncwarp();
    }

    // ---- merge the warps of this CTA
    if (lane == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            wm[warp][h] = m[h];
            wl[warp][h] = l[h];
        }
    }
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < DPL; ++e) wacc[warp][h][lane * DPL + e] = acc[h][e];
    __syncthreads();

    const int n_heads = p.n_heads;
    for (int i = threadIdx.x; i < G * HD; i += kAttnThreads) {
        const int h = i / HD, d = i - h * HD;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, wm[w][h]);
        float Ls = 0.f, A = 0.f;
#pragma unroll
        for (int w = 0; w < kAttnWarps; ++w) {
            const float f = (wm[w][h] == -INFINITY) ? 0.f : exp2f(wm[w][h] - M);
            Ls += wl[w][h] * f;
            A += wacc[w][h][d] * f;
        }
        const int hg = g * G + h;
        if (n_active == 1) {
            p.out[((size_t)b * n_heads + hg) * HD + d] = __float2half_rn(A / Ls);
        } else {
            const size_t slot = ((size_t)b * n_heads + hg) * p.nsplit + s;
            p.pacc[slot * HD + d] = A;
            if (d == 0) {
                p.pm[slot] = M;
                p.pl[slot] = Ls;
            }
        }
    }
    if (n_active == 1) return;

    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const int ticket = atomicAdd(&p.tickets[b * p.n_kv + g], 1);
        last_flag = (ticket == n_active - 1);
    }
    __syncthreads();
    if (!last_flag) return;
    __threadfence();
    // merge: per-split weights exp2(m_k - M) / L into shared memory (one warp per head), then
    // every thread sums float4 chunks of the partial outputs with independent loads
    __shared__ float sw[G][kMaxSplit];
    for (int h = warp; h < G; h += kAttnWarps) {
        const size_t base = ((size_t)b * n_heads + g * G + h) * p.nsplit;
        float M = -INFINITY;
        for (int k = lane; k < n_active; k += 32) M = fmaxf(M, __ldcg(p.pm + base + k));
#pragma unroll
        for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float Ls = 0.f;
        for (int k = lane; k < n_active; k += 32) {
            const float f = exp2f(__ldcg(p.pm + base + k) - M);
            sw[h][k] = f;
            Ls += f * __ldcg(p.pl + base + k);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
        const float inv = 1.0f / Ls;
        __syncwarp();
        for (int k = lane; k < n_active; k += 32) sw[h][k] *= inv;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < G * HD / 4; i += kAttnThreads) {
        const int h = i / (HD / 4), d4 = i - h * (HD / 4);
        const size_t base = ((size_t)b * n_heads + g * G + h) * p.nsplit;
        const float4* src = reinterpret_cast<const float4*>(p.pacc) + base * (HD / 4) + d4;
        float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
        int k = 0;
        for (; k + 8 <= n_active; k += 8) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = __ldcg(src + (size_t)(k + u) * (HD / 4));
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const float w = sw[h][k + u];
                A.x = fmaf(w, v[u].x, A.x); A.y = fmaf(w, v[u].y, A.y);
                A.z = fmaf(w, v[u].z, A.z); A.w = fmaf(w, v[u].w, A.w);
            }
        }
        for (; k < n_active; ++k) {
            const float4 v = __ldcg(src + (size_t)k * (HD / 4));
            const float w = sw[h][k];
            A.x = fmaf(w, v.x, A.x); A.y = fmaf(w, v.y, A.y);
            A.z = fmaf(w, v.z, A.z); A.w = fmaf(w, v.w, A.w);
        }
        __half* o = p.out + ((size_t)b * n_heads + g * G + h) * HD + d4 * 4;
        *reinterpret_cast<__half2*>(o) = __floats2half2_rn(A.x, A.y);
        *reinterpret_cast<__half2*>(o + 2) = __floats2half2_rn(A.z, A.w);
    }
    if (threadIdx.x == 0) p.tickets[b * p.n_kv + g] = 0;   // re-arm for the next call
}

struct Layout {
    int nsplit, spb;
    size_t tickets_off, pm_off, pl_off, pacc_off, total;
};

Layout layout(int64_t batch, int n_heads, int n_kv, int head_dim, int64_t maxb, int sms) {
    Layout lo = {};
    // Split the block table so that a full-capacity batch gives several CTAs per SM.
    const int64_t pairs = batch * n_kv;
    const int64_t target = 8ll * sms;
    int64_t spb = (maxb * pairs + target - 1) / target;
    if (spb < 4) spb = 4;
    if (spb > maxb) spb = maxb;
    if (spb < 1) spb = 1;
    if ((maxb + spb - 1) / spb > kMaxSplit) spb = (maxb + kMaxSplit - 1) / kMaxSplit;
    lo.spb = (int)spb;
    lo.nsplit = (int)((maxb + spb - 1) / spb);
    auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
    size_t off = 0;
    lo.tickets_off = off;
    off = al(off + (size_t)pairs * sizeof(int));
    lo.pm_off = off;
    off = al(off + (size_t)batch * n_heads * lo.nsplit * sizeof(float));
    lo.pl_off = off;
    off = al(off + (size_t)batch * n_heads * lo.nsplit * sizeof(float));
    lo.pacc_off = off;
    off = al(off + (size_t)batch * n_heads * lo.nsplit * head_dim * sizeof(float));
    lo.total = off;
    return lo;
}

template <int HD, int G>
cudaError_t launch_hg(const AParams& p, int batch, cudaStream_t s, bool pdl) {
    dim3 grid(p.nsplit, p.n_kv, batch);
    return launch(attn_split_kernel<HD, G>, grid, dim3(kAttnThreads), 0, s, pdl, p,
                  device_error_record());
}

template <int HD>
cudaError_t launch_h(const AParams& p, int G, int batch, cudaStream_t s, bool pdl) {
    switch (G) {
        case 1: return launch_hg<HD, 1>(p, batch, s, pdl);
        case 2: return launch_hg<HD, 2>(p, batch, s, pdl);
        case 4: return launch_hg<HD, 4>(p, batch, s, pdl);
        case 8: return launch_hg<HD, 8>(p, batch, s, pdl);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

size_t attn_workspace_bytes(int64_t batch, int n_heads, int n_kv_heads, int head_dim,
                            int block_size, int64_t max_blocks_per_seq) {
    (void)block_size;
    if (batch <= 0 || n_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 || max_blocks_per_seq <= 0)
        return 0;
    return layout(batch, n_heads, n_kv_heads, head_dim, max_blocks_per_seq, num_sms()).total;
}

int attn_launch(const AttnArgs& a, cudaStream_t s, bool pdl) {
    QL_REQUIRE(a.q && a.k_pool && a.v_pool && a.block_tables && a.out && a.workspace,
               "attention: null pointer");
    QL_REQUIRE(a.context_lens || a.positions, "attention: need context lengths or positions");
    QL_REQUIRE(a.head_dim == 64 || a.head_dim == 128, "attention: head_dim must be 64 or 128");
    QL_REQUIRE(a.block_size == kBS, "attention: block_size must be 16");
    QL_REQUIRE(a.n_kv_heads > 0 && a.n_heads % a.n_kv_heads == 0, "attention: n_heads % n_kv_heads != 0");
    const int G = a.n_heads / a.n_kv_heads;
    QL_REQUIRE(G == 1 || G == 2 || G == 4 || G == 8, "attention: GQA group must be 1, 2, 4 or 8");
    QL_REQUIRE(a.batch >= 1 && a.batch <= 65535, "attention: batch out of range");
    QL_REQUIRE(a.max_blocks_per_seq >= 1 && a.max_blocks_per_seq * kBS < (1ll << 31),
               "attention: bad max_blocks_per_seq");
    QL_REQUIRE(a.num_blocks >= 1, "attention: bad num_blocks");
    const Layout lo = layout(a.batch, a.n_heads, a.n_kv_heads, a.head_dim, a.max_blocks_per_seq, num_sms());
    if (a.workspace_bytes < lo.total)
        return set_error(QL_EINVAL, "attention: workspace too small (need " + std::to_string(lo.total) + " bytes)");
    QL_REQUIRE(((reinterpret_cast<uintptr_t>(a.k_pool) | reinterpret_cast<uintptr_t>(a.v_pool)) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(a.out) & 3) == 0 && (reinterpret_cast<uintptr_t>(a.q) & 1) == 0,
               "attention: K/V pools must be 16-byte aligned, the output 4-byte aligned");
    if (!device_error_record()) return set_error(QL_ECUDA, "attention: no device error record");
    AParams p = {};
    p.q = a.q;
    p.k_pool = a.k_pool;
    p.v_pool = a.v_pool;
    p.block_tables = a.block_tables;
    p.context_lens = a.context_lens;
    p.positions = a.positions;
    p.active = a.active;
    p.n_heads = a.n_heads;
    p.n_kv = a.n_kv_heads;
    p.maxb = (int)a.max_blocks_per_seq;
    p.num_blocks = a.num_blocks;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.out = a.out;
    char* ws = static_cast<char*>(a.workspace);
    p.tickets = reinterpret_cast<int*>(ws + lo.tickets_off);
    p.pm = reinterpret_cast<float*>(ws + lo.pm_off);
    p.pl = reinterpret_cast<float*>(ws + lo.pl_off);
    p.pacc = reinterpret_cast<float*>(ws + lo.pacc_off);
    p.nsplit = lo.nsplit;
    p.spb = lo.spb;
    p.prefetch = a.context_lens == nullptr ? 1 : 0;
    cudaError_t e = a.head_dim == 128 ? launch_h<128>(p, G, a.batch, s, pdl)
                                      : launch_h<64>(p, G, a.batch, s, pdl);
    if (e != cudaSuccess) return cuda_error(e, "attention launch");
    return QL_OK;
}

}  // namespace ql

extern "C" size_t ql_paged_attn_workspace_bytes(int64_t batch, int n_heads, int n_kv_heads,
                                                int head_dim, int block_size,
                                                int64_t max_blocks_per_seq) {
    return ql::attn_workspace_bytes(batch, n_heads, n_kv_heads, head_dim, block_size,
                                    max_blocks_per_seq);
}

extern "C" int ql_paged_attn_decode(const void* d_q, const void* d_k_pool, const void* d_v_pool,
                                    const int32_t* d_block_tables, const int32_t* d_context_lens,
                                    int64_t batch, int n_heads, int n_kv_heads, int head_dim,
                                    int block_size, int64_t max_blocks_per_seq, int64_t num_blocks,
                                    float scale, void* d_out, void* d_workspace,
                                    size_t workspace_bytes, void* stream) {
    using namespace ql;
    QL_REQUIRE(d_context_lens, "ql_paged_attn_decode: null context lengths");
    AttnArgs a = {};
    a.q = static_cast<const __half*>(d_q);
    a.k_pool = static_cast<const __half*>(d_k_pool);
    a.v_pool = static_cast<const __half*>(d_v_pool);
    a.block_tables = d_block_tables;
    a.context_lens = d_context_lens;
    a.batch = (int)batch;
    a.n_heads = n_heads;
    a.n_kv_heads = n_kv_heads;
    a.head_dim = head_dim;
    a.block_size = block_size;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.scale = scale;
    a.out = static_cast<__half*>(d_out);
    a.workspace = d_workspace;
    a.workspace_bytes = workspace_bytes;
    if (batch < 1 || batch > 65535) return set_error(QL_EINVAL, "ql_paged_attn_decode: batch out of range");
    return attn_launch(a, static_cast<cudaStream_t>(stream), true);
}

// ------------------------------------------------------------------ no-allocation variant
// Some callers cannot allocate device memory for the split-K workspace: a plugin running
// inside a host application that owns every byte of device memory through its own pool (a raw
// cudaMalloc would bypass that pool's accounting or exceed its budget), or a latency-critical
// loop that must not pay for cudaMalloc / cudaFree, which can synchronise the whole device.
// ql_paged_attn_decode_noalloc serves them from a fixed scratch array that lives in the
// library image itself; every GPU that loads the library holds it until the process exits.
#include <map>
#include <mutex>

namespace ql {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)8 << 20;   // 8 MiB per device
static __device__ __align__(256) unsigned char g_attn_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
std::map<int, void*> g_noalloc_addr;

// Device address of the scratch array on the current device. In host code the array's name is
// only a host-side stand-in, so the address is looked up once per device, with that device
// current, and cached.
int noalloc_scratch_address(void** out) {
    int dev = 0;
    QL_TRY_CUDA(cudaGetDevice(&dev));
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    auto it = g_noalloc_addr.find(dev);
    if (it == g_noalloc_addr.end()) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_attn_noalloc_scratch);
        if (e != cudaSuccess) return cuda_error(e, "ql_paged_attn_decode_noalloc: cudaGetSymbolAddress");
        it = g_noalloc_addr.emplace(dev, p).first;
    }
    *out = it->second;
    return QL_OK;
}

template <int HD, int G>
cudaError_t launch_hg_err(const AParams& p, int batch, cudaStream_t s, DevError* err) {
    dim3 grid(p.nsplit, p.n_kv, batch);
    return launch(attn_split_kernel<HD, G>, grid, dim3(kAttnThreads), 0, s, true, p, err);
}

template <int HD>
cudaError_t launch_h_err(const AParams& p, int G, int batch, cudaStream_t s, DevError* err) {
    switch (G) {
        case 1: return launch_hg_err<HD, 1>(p, batch, s, err);
        case 2: return launch_hg_err<HD, 2>(p, batch, s, err);
        case 4: return launch_hg_err<HD, 4>(p, batch, s, err);
        case 8: return launch_hg_err<HD, 8>(p, batch, s, err);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace
}  // namespace ql

extern "C" int ql_paged_attn_decode_noalloc(const void* d_q, const void* d_k_pool, const void* d_v_pool,
                                            const int32_t* d_block_tables,
                                            const int32_t* d_context_lens, int64_t batch,
                                            int n_heads, int n_kv_heads, int head_dim,
                                            int block_size, int64_t max_blocks_per_seq,
                                            int64_t num_blocks, float scale, void* d_out,
                                            void* stream) {
    using namespace ql;
    QL_REQUIRE(d_q && d_k_pool && d_v_pool && d_block_tables && d_context_lens && d_out,
               "ql_paged_attn_decode_noalloc: null pointer");
    QL_REQUIRE(head_dim == 64 || head_dim == 128, "ql_paged_attn_decode_noalloc: head_dim must be 64 or 128");
    QL_REQUIRE(block_size == kBS, "ql_paged_attn_decode_noalloc: block_size must be 16");
    QL_REQUIRE(n_kv_heads > 0 && n_heads > 0 && n_heads % n_kv_heads == 0,
               "ql_paged_attn_decode_noalloc: n_heads % n_kv_heads != 0");
    const int G = n_heads / n_kv_heads;
    QL_REQUIRE(G == 1 || G == 2 || G == 4 || G == 8, "ql_paged_attn_decode_noalloc: GQA group must be 1, 2, 4 or 8");
    QL_REQUIRE(batch >= 1 && batch <= 65535, "ql_paged_attn_decode_noalloc: batch out of range");
    QL_REQUIRE(max_blocks_per_seq >= 1 && max_blocks_per_seq * kBS < (1ll << 31),
               "ql_paged_attn_decode_noalloc: bad max_blocks_per_seq");
    QL_REQUIRE(num_blocks >= 1, "ql_paged_attn_decode_noalloc: bad num_blocks");
    const Layout lo = layout(batch, n_heads, n_kv_heads, head_dim, max_blocks_per_seq, num_sms());
    if (lo.total > kNoAllocScratchBytes)
        return set_error(QL_EINVAL, "ql_paged_attn_decode_noalloc: this shape needs " +
                                        std::to_string(lo.total) + " bytes of split-K scratch, more than the " +
                                        std::to_string(kNoAllocScratchBytes) +
                                        " bytes built into the library; use ql_paged_attn_decode with a workspace");
    void* scratch = nullptr;
    if (int rc = noalloc_scratch_address(&scratch)) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the split tickets must start at zero; the array keeps whatever the last call left
    QL_TRY_CUDA(cudaMemsetAsync(static_cast<char*>(scratch) + lo.tickets_off, 0,
                                (size_t)batch * n_kv_heads * sizeof(int), s));
    AParams p = {};
    p.q = static_cast<const __half*>(d_q);
    p.k_pool = static_cast<const __half*>(d_k_pool);
    p.v_pool = static_cast<const __half*>(d_v_pool);
    p.block_tables = d_block_tables;
    p.context_lens = d_context_lens;
    p.positions = nullptr;
    p.active = nullptr;
    p.n_heads = n_heads;
    p.n_kv = n_kv_heads;
    p.maxb = (int)max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.out = static_cast<__half*>(d_out);
    char* ws = static_cast<char*>(scratch);
    p.tickets = reinterpret_cast<int*>(ws + lo.tickets_off);
    p.pm = reinterpret_cast<float*>(ws + lo.pm_off);
    p.pl = reinterpret_cast<float*>(ws + lo.pl_off);
    p.pacc = reinterpret_cast<float*>(ws + lo.pacc_off);
    p.nsplit = lo.nsplit;
    p.spb = lo.spb;
    p.prefetch = 0;
    // out-of-range indices are skipped; they are recorded only if this device already has an
    // error record (this path never creates one, since that would allocate)
    DevError* err = device_error_record_existing();
    const cudaError_t e = head_dim == 128 ? launch_h_err<128>(p, G, (int)batch, s, err)
                                          : launch_h_err<64>(p, G, (int)batch, s, err);
    if (e != cudaSuccess) return cuda_error(e, "ql_paged_attn_decode_noalloc launch");
    return QL_OK;
}
