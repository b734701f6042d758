// Paged split-K GQA decode attention over an f16 block pool.
//
// [FK] ferrum-kernels cuda_decode.rs: launch_paged_decode_attention / attention_paged (16-token
// blocks, block table, valid length = current length + 1, scale 1/sqrt(hd)) and the split-K
// flash-decode phase 1 + reduce; [IL] inferencelayer cuda_llm.rs CudaQwen3::step
// (attn_partial + attn_reduce over per-(head, chunk) running max / sum / weighted V).
//
// out[b][h] = sum_t softmax_t(q[b][h] . k[g][t] * scale) v[g][t], g = h / (n_heads / n_kv).
//
// Design (GB300): one CTA per (split, kv head, sequence), 8 warps at batch 1-2, else 4. The CTA
// handles the whole GQA group of its kv head, so each K/V byte is read from HBM once and used
// by all G query heads. A warp takes 16-token blocks in turn, staged in shared memory with
// cp.async (double-buffered); S = Q K^T and O += P V run on mma.sync (ldmatrix, .trans for V)
// with an online softmax in the exp2 domain (scores pre-scaled by scale * log2 e). The warps'
// states are merged in shared memory; with one split the CTA writes the output. Otherwise the
// splits are merged in one of two forms:
//  * ticket (default): each CTA writes its partial to global memory, and the last CTA of its
//    (sequence, kv head) - found with an atomic ticket, no waiting - merges all partials and
//    re-arms the ticket. Most CTAs exit right after their ticket, so the next kernel's CTAs
//    find their SMs free early;
//  * cluster (selectable; batch 1-2, up to 16 splits, when the device can hold one cluster per
//    (sequence, kv head) at once): the splits of a (sequence, kv head) are one thread-block
//    cluster; each CTA keeps its (m, l, acc) partial in shared memory, and after a cluster
//    barrier every CTA merges a slice of the outputs, reading the others' partials through
//    distributed shared memory; a second barrier keeps the partials alive until all reads are
//    done. Every CTA then lives until the merge ends, and the decode step measured slower.
#include <cuda_fp16.h>
#include <math.h>

#include <atomic>
#include <cstdlib>
#include <map>
#include <mutex>
#include <set>

#include "ql_internal.h"
#include "ql_kvq_rec.cuh"

namespace ql {
namespace {

// warps per CTA: 8 at batch 1-2 (16-block splits, every block of a warp staged before the wait,
// half the splits to merge), else 4 (more CTAs per SM for long batched contexts)
constexpr int attn_warps(int64_t batch) { return batch <= 2 ? 8 : 4; }
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
    NextWeights next;   // weights of the following kernel, prefetched into L2
    // fused qk-norm + RoPE + KV append (decode step): q and the new K/V come from the f32 qkv
    // projection instead of q; the CTA whose split holds the new position writes K/V to the pool
    const float* qkv;
    const float* q_norm;
    const float* k_norm;
    const float* cos_t;
    const float* sin_t;
    float eps;
    long long max_position;
    __half* kw;
    __half* vw;
    // quantised pool (KQ kernels): one record per (block, kv head), keys q8_0 and values q5_1
    // (ql_kvq_rec.cuh); read by the attention, written by the fused append
    uint8_t* kvq;
    unsigned long long* trace;   // optional stamps of the CTAs with linear index < trace_ctas
    int trace_ctas;
};

__device__ __forceinline__ void attn_stamp(unsigned long long* tr, int i) {
    if (tr != nullptr && threadIdx.x == 0) {
        unsigned long long t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        tr[i] = t;
    }
}

// Physical block of logical block lb of sequence b, or -1 if the table entry is out of range.
__device__ __forceinline__ int bt_row_phys(const AParams& p, int b, int lb) {
    const int phys = p.block_tables[(size_t)b * p.maxb + lb];
    return (phys >= 0 && phys < p.num_blocks) ? phys : -1;
}

// What one lane needs of a norm weight and of the rotation table row for warp_norm_rope:
// elements i and i + HD/2 for i = lane, lane + 32, ... (loaded before the kernel waits on its
// predecessor: weights and tables are constants of the step).
template <int HD>
struct RopeLane {
    static constexpr int PER = HD / 64;
    float wa[PER], wb[PER], c[PER], s[PER];
};
template <int HD>
__device__ __forceinline__ RopeLane<HD> rope_lane(const float* w, const float* cos_row, const float* sin_row,
                                                  int lane) {
    RopeLane<HD> r;
#pragma unroll
    for (int k = 0; k < RopeLane<HD>::PER; ++k) {
        const int i = lane + 32 * k;
        r.wa[k] = __ldg(w + i);
        r.wb[k] = __ldg(w + i + HD / 2);
        r.c[k] = __ldg(cos_row + i);
        r.s[k] = __ldg(sin_row + i);
    }
    return r;
}

// RMSNorm over one head (weight w) and NeoX rotation at table row `pos`, by one warp:
// lane handles the pairs (i, i + HD/2) for i = lane, lane + 32, ...; writes f16 to dst.
template <int HD>
__device__ __forceinline__ void warp_norm_rope(const float* src, const RopeLane<HD>& rl, float eps, __half* dst,
                                               int lane) {
    constexpr int H2 = HD / 2, PER = RopeLane<HD>::PER;
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
        const float a = xa[k] * r * rl.wa[k], bb = xb[k] * r * rl.wb[k];
        dst[i] = __float2half_rn(a * rl.c[k] - bb * rl.s[k]);
        dst[i + H2] = __float2half_rn(a * rl.s[k] + bb * rl.c[k]);
    }
}

// The same normalisation and rotation with the f32 results kept in registers: out[k] is
// dimension lane + 32 k (the layout of the warp-level KV quantisers).
template <int HD>
__device__ __forceinline__ void warp_norm_rope_vals(const float* src, const RopeLane<HD>& rl, float eps, int lane,
                                                    float (&out)[HD / 32]) {
    constexpr int H2 = HD / 2, PER = RopeLane<HD>::PER;
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
        const float a = xa[k] * r * rl.wa[k], bb = xb[k] * r * rl.wb[k];
        out[k] = a * rl.c[k] - bb * rl.s[k];
        out[k + PER] = a * rl.s[k] + bb * rl.c[k];
    }
}

__device__ __forceinline__ float2 h2f(uint32_t u) {
    __half2 h;
    *reinterpret_cast<uint32_t*>(&h) = u;
    return __half22float2(h);
}

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Thread-block cluster primitives (PTX): a full cluster barrier (every thread of every CTA
// arrives; release/acquire order the shared-memory partials), the cluster address of a shared
// variable in the CTA of rank r, and loads through it.
__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_addr(uint32_t cta_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(cta_addr), "r"(rank));
    return r;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
    return v;
}

// CL: the splits of a (sequence, kv head) form one cluster (grid x = cluster x = nsplit) and are
// merged through distributed shared memory; otherwise by the ticket.
// KQ: the pool is quantised (keys q8_0, values q5_1, one record of 29 HD bytes per (block, kv
// head), ql_kvq_rec.cuh): a warp stages its blocks' records (double-buffered) and decodes each
// into one pair of f16 K / V tiles just before its MMAs; the fused append quantises the new rows.
template <int HD, int G, int NW, bool CL, bool KQ = false>
__global__ void __launch_bounds__(NW * 32) attn_split_kernel(AParams p, DevError* err) {
    constexpr int kAttnWarps = NW, kAttnThreads = NW * 32;
    constexpr int KSTEPS = HD / 16;           // k-steps of the Q.K^T MMA
    constexpr int NT = HD / 8;                // 8-dim output tiles of the P.V MMA
    constexpr int PITCH = HD * 2 + 16;        // bytes per staged K/V row (padded: conflict-free ldmatrix)
    constexpr int TILE = kBS * PITCH;         // one staged 16-key K or V tile
    constexpr int CHUNKS = HD * 2 / 16;       // 16-byte chunks per K/V row
    constexpr int REC = Kvq<HD>::BYTES;       // one quantised record (KQ)
    constexpr int WBYTES = KQ ? 2 * REC + 2 * TILE : 4 * TILE;   // shared memory per warp
    extern __shared__ __align__(16) unsigned char asmem[];   // staged tiles, later the merge buffers
    __shared__ float wm[kAttnWarps][G], wl[kAttnWarps][G];
    __shared__ int last_flag;

    const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // Fused decode-step form (qkv set): the context length and the K/V of earlier positions are
    // final before this kernel starts (every kernel of the step triggers its successor only
    // after its own wait, so everything two launches back has completed), and the new
    // position's row is appended by this kernel: the first K/V tiles are staged before the
    // wait and the new row is patched into them. Otherwise q, K/V or the lengths may come from
    // the previous kernel: wait first.
    const bool fused = p.qkv != nullptr;
    const int lin = (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
    unsigned long long* tr = (p.trace != nullptr && lin < p.trace_ctas) ? p.trace + (size_t)lin * 8 : nullptr;
    attn_stamp(tr, 0);
    l2_prefetch_share(p.next.ptr[0], p.next.bytes[0]);
    l2_prefetch_share(p.next.ptr[1], p.next.bytes[1]);
    if (!fused) {
        pdl_wait();
        pdl_trigger();
    }
    // The CTA's first loads, in flight together (one round trip instead of a chain of three):
    // the slot's activity, its length, and the block-table entries of this warp's first two
    // blocks (a split's first block, s * spb, does not depend on the length; entries are read
    // only inside the table's row).
    const int32_t* bt = p.block_tables + (size_t)b * p.maxb;
    const int e0 = s * p.spb + warp;
    const int act = p.active ? p.active[b] : 1;
    const int L = p.context_lens ? p.context_lens[b] : p.positions[b] + 1;
    const int pre0 = e0 < p.maxb ? bt[e0] : -1;
    const int pre1 = e0 + kAttnWarps < p.maxb ? bt[e0 + kAttnWarps] : -1;
    if (act == 0) return;
    if (L <= 0) return;   // idle slot
    if (L > p.maxb * kBS) {
        if (s == 0 && threadIdx.x == 0) record_device_error(err, kErrAttnLength, b, L);
        return;
    }
    const int nblocks = (L + kBS - 1) / kBS;
    const int n_active = (nblocks + p.spb - 1) / p.spb;
    if (s >= n_active) {
        // an idle split of a cluster still takes part in both of its barriers (the decision is
        // the same in every CTA of the cluster: one (sequence, kv head), one n_active)
        if (CL && n_active > 1) {
            cluster_barrier();
            cluster_barrier();
        }
        return;
    }
    const int blk0 = s * p.spb;
    const int blk1 = min(nblocks, blk0 + p.spb);
    const int pos = L - 1, lblk = pos / kBS, kp = pos % kBS;

    // f16: [buffer][K | V] tiles; KQ: [buffer] records, then one decoded K | V tile pair
    unsigned char* wtiles = asmem + (size_t)warp * WBYTES;
    const uint32_t wtiles_s = static_cast<uint32_t>(__cvta_generic_to_shared(wtiles));
    const int nb_w = blk1 - blk0 > warp ? (blk1 - blk0 - warp + kAttnWarps - 1) / kAttnWarps : 0;

    // stage block i of this warp into buffer (i & 1) with 16-byte asynchronous copies (blocks 0
    // and 1: their table entries were loaded with the length)
    auto stage = [&](int i) -> bool {
        const int blk = blk0 + warp + kAttnWarps * i;
        const int phys = i == 0 ? pre0 : (i == 1 ? pre1 : bt[blk]);
        bool ok = phys >= 0 && phys < p.num_blocks;
        if (!ok) {
            if (lane == 0) record_device_error(err, kErrAttnBlock, (long long)b * p.maxb + blk, phys);
        } else if (KQ) {
            const unsigned char* src = p.kvq + ((size_t)phys * p.n_kv + g) * REC;
            const uint32_t dst = wtiles_s + (uint32_t)((i & 1) * REC);
            const unsigned long long pol = l2_evict_first();
            for (int c = lane; c < REC / 16; c += 32)
                asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst + c * 16),
                             "l"(src + c * 16), "l"(pol) : "memory");
        } else {
            const __half* ksrc = p.k_pool + ((size_t)phys * p.n_kv + g) * kBS * HD;
            const __half* vsrc = p.v_pool + ((size_t)phys * p.n_kv + g) * kBS * HD;
            const uint32_t kd = wtiles_s + (uint32_t)((i & 1) * 2 * TILE), vd = kd + TILE;
            const unsigned long long pol = l2_evict_first();   // the context is read once per step
            for (int c = lane; c < kBS * CHUNKS; c += 32) {
                const int row = c / CHUNKS, col = c - row * CHUNKS;
                asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(kd + row * PITCH + col * 16),
                             "l"(ksrc + row * HD + col * 8), "l"(pol) : "memory");
                asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(vd + row * PITCH + col * 16),
                             "l"(vsrc + row * HD + col * 8), "l"(pol) : "memory");
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        return ok;
    };
    // both buffers of the warp in flight from the start (blocks 0 and 1; an empty group when the
    // warp has one block): in the fused form before the wait
    bool vbuf[2] = {false, false};
    auto stage_first = [&]() {
        if (nb_w > 0) vbuf[0] = stage(0);
        if (nb_w > 1) vbuf[1] = stage(1);
        else asm volatile("cp.async.commit_group;" ::: "memory");
    };
    const bool pos_ok = pos < p.max_position;
    RopeLane<HD> rq, rk;
    if (fused) {
        stage_first();
        const float* cr = p.cos_t + (size_t)(pos_ok ? pos : 0) * (HD / 2);
        const float* sr = p.sin_t + (size_t)(pos_ok ? pos : 0) * (HD / 2);
        rq = rope_lane<HD>(p.q_norm, cr, sr, lane);
        if (warp == 0) rk = rope_lane<HD>(p.k_norm, cr, sr, lane);
        pdl_wait();
        pdl_trigger();
        attn_stamp(tr, 1);
    }

    // Q as the A operand of S = Q K^T: rows = the G heads of this kv head (rows >= G and the
    // fragment's rows g + 8 are zero padding); lane (gq, tq) holds dims 16 kk + 2 tq (+8).
    const int gq = lane >> 2, tq = lane & 3;
    const bool hv = gq < G;
    uint32_t qa[KSTEPS][2];
    __shared__ __align__(16) __half qs[G][HD];
    __shared__ __align__(16) __half knew[HD];   // the appended K row (normed, rotated) and V row
    __shared__ __align__(16) __half vnew[HD];
    const __half* qsrc;
    if (fused) {
        // normalise + rotate the G query heads here; the CTA holding the new position's block
        // also normalises + rotates the new key and appends K and V
        const float* src = p.qkv + (size_t)b * (p.n_heads + 2 * p.n_kv) * HD;
        if (!pos_ok && s == 0 && threadIdx.x == 0) record_device_error(err, kErrRopePosition, b, pos);
        for (int h = warp; h < G; h += kAttnWarps)
            warp_norm_rope<HD>(src + (size_t)(g * G + h) * HD, rq, p.eps, qs[h], lane);
        if (pos_ok && lblk >= blk0 && lblk < blk1 && warp < 2) {
            const int phys = bt_row_phys(p, b, lblk);
            if (phys < 0) {
                if (lane == 0) record_device_error(err, kErrRopeBlock, (long long)b * p.maxb + lblk, phys);
            } else {
                const size_t off = (((size_t)phys * p.n_kv + g) * kBS + kp) * HD;
                if (KQ) {
                    // quantise the new rows into the record (keys q8_0 from the rotated f32 K,
                    // values q5_1 from the f32 V); knew / vnew get them as the tiles decode them
                    uint8_t* rec = p.kvq + ((size_t)phys * p.n_kv + g) * REC;
                    float xr[HD / 32];
                    bool ok;
                    if (warp == 0) {
                        warp_norm_rope_vals<HD>(src + (size_t)(p.n_heads + g) * HD, rk, p.eps, lane, xr);
                        ok = kvq_put_k_row<HD>(xr, rec, kp, lane, knew);
                    } else {
                        const float* vs = src + (size_t)(p.n_heads + p.n_kv + g) * HD;
#pragma unroll
                        for (int k = 0; k < HD / 32; ++k) xr[k] = __ldcg(vs + lane + 32 * k);
                        ok = kvq_put_v_row<HD>(xr, rec, kp, lane, vnew);
                    }
                    if (!ok && lane == 0) record_device_error(err, kErrKvOverflow, (long long)b * p.maxb + lblk, kp);
                } else if (warp == 0) {
                    warp_norm_rope<HD>(src + (size_t)(p.n_heads + g) * HD, rk, p.eps, knew, lane);
                    __syncwarp();
                    for (int i = lane; i < HD / 8; i += 32)
                        reinterpret_cast<uint4*>(p.kw + off)[i] = reinterpret_cast<const uint4*>(knew)[i];
                } else {
                    const float* vs = src + (size_t)(p.n_heads + p.n_kv + g) * HD;
                    for (int i = lane; i < HD; i += 32) {
                        const __half v = __float2half_rn(vs[i]);
                        vnew[i] = v;
                        p.vw[off + i] = v;
                    }
                }
            }
        }
        __threadfence_block();
        __syncthreads();
        attn_stamp(tr, 2);
        qsrc = &qs[0][0];
    } else {
        qsrc = p.q + ((size_t)b * p.n_heads + g * G) * HD;
    }
    {
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(qsrc + (size_t)(hv ? gq : 0) * HD);
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk) {
            qa[kk][0] = hv ? qrow[8 * kk + tq] : 0u;
            qa[kk][1] = hv ? qrow[8 * kk + 4 + tq] : 0u;
        }
    }
    float o[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float mrow = -INFINITY, lrow = 0.f;
    if (!fused) stage_first();
    for (int i = 0; i < nb_w; ++i) {
        // groups committed so far: blocks 0 .. i + 1 (one per block, empty past the end); block i
        // has landed when at most one group is pending
        asm volatile("cp.async.wait_group 1;" ::: "memory");
        __syncwarp();
        const bool vcur = vbuf[i & 1];
        const int blk = blk0 + warp + kAttnWarps * i;
        const int nt = min(kBS, L - blk * kBS);      // valid keys in this block
        // the f16 tiles this block is read from: its staging buffer, or (KQ) the decoded pair
        const int tbuf = KQ ? 2 * REC : (i & 1) * 2 * TILE;
        if (KQ && vcur) {
            kvq_decode_tile<HD>(wtiles + (size_t)(i & 1) * REC, wtiles + tbuf, wtiles + tbuf + TILE, PITCH, lane);
            __syncwarp();
        }
        if (vcur && fused && blk == lblk) {
            // the new row: staged (possibly) before it was appended, so patch it in
            unsigned char* kt = wtiles + tbuf;
            if (lane < CHUNKS)
                *reinterpret_cast<uint4*>(kt + kp * PITCH + lane * 16) = reinterpret_cast<const uint4*>(knew)[lane];
            else if (lane < 2 * CHUNKS)
                *reinterpret_cast<uint4*>(kt + TILE + kp * PITCH + (lane - CHUNKS) * 16) =
                    reinterpret_cast<const uint4*>(vnew)[lane - CHUNKS];
            __syncwarp();
        }
        if (vcur) {
            unsigned char* vtile = wtiles + tbuf + TILE;
            if (nt < kBS) {
                // keys past the context: their P is 0, but a stale V row must not be NaN/Inf
                for (int c = lane; c < (kBS - nt) * CHUNKS; c += 32) {
                    const int row = nt + c / CHUNKS, col = c % CHUNKS;
                    *reinterpret_cast<uint4*>(vtile + row * PITCH + col * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                __syncwarp();
            }
            const uint32_t ks = wtiles_s + (uint32_t)tbuf, vs = ks + TILE;
            // ---- S = Q K^T for the 16 keys (two 8-key tiles)
            float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
            const int lm = lane >> 3, lr = lane & 7;
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
                uint32_t b0, b1, b2, b3;
                const uint32_t addr = ks + (uint32_t)(((lm >> 1) * 8 + lr) * PITCH + (16 * kk + (lm & 1) * 8) * 2);
                asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                             : "=r"(b0), "=r"(b1), "=r"(b2), "=r"(b3) : "r"(addr));
                mma_f16(s0, qa[kk][0], 0u, qa[kk][1], 0u, b0, b1);
                mma_f16(s1, qa[kk][0], 0u, qa[kk][1], 0u, b2, b3);
            }
            // ---- online softmax of head row gq over the block's keys (exp2 domain)
            const int k0 = 2 * tq;
            const float x0 = k0 < nt ? s0[0] * p.scale_log2 : -INFINITY;
            const float x1 = k0 + 1 < nt ? s0[1] * p.scale_log2 : -INFINITY;
            const float x2 = k0 + 8 < nt ? s1[0] * p.scale_log2 : -INFINITY;
            const float x3 = k0 + 9 < nt ? s1[1] * p.scale_log2 : -INFINITY;
            float mb = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
            mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
            mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
            const float mn = fmaxf(mrow, mb);
            const float alpha = exp2f(mrow - mn);
            const float p0 = exp2f(x0 - mn), p1 = exp2f(x1 - mn), p2 = exp2f(x2 - mn), p3 = exp2f(x3 - mn);
            float ls = (p0 + p1) + (p2 + p3);
            ls += __shfl_xor_sync(0xffffffffu, ls, 1);
            ls += __shfl_xor_sync(0xffffffffu, ls, 2);
            lrow = lrow * alpha + ls;
            mrow = mn;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                o[n][0] *= alpha;
                o[n][1] *= alpha;
            }
            const __half2 pa0 = __floats2half2_rn(p0, p1), pa1 = __floats2half2_rn(p2, p3);
            const uint32_t ua0 = *reinterpret_cast<const uint32_t*>(&pa0);
            const uint32_t ua1 = *reinterpret_cast<const uint32_t*>(&pa1);
            // ---- O += P V (V^T fragments by transposing ldmatrix)
#pragma unroll
            for (int pp = 0; pp < NT / 2; ++pp) {
                uint32_t r0, r1, r2, r3;
                const uint32_t addr = vs + (uint32_t)(((lm & 1) * 8 + lr) * PITCH + (16 * pp + (lm >> 1) * 8) * 2);
                asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                             : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
                mma_f16(o[2 * pp], ua0, 0u, ua1, 0u, r0, r1);
                mma_f16(o[2 * pp + 1], ua0, 0u, ua1, 0u, r2, r3);
            }
        }
        __syncwarp();   // every lane is done with buffer i & 1: block i + 2 may land there
        if (i + 2 < nb_w) vbuf[i & 1] = stage(i + 2);
        else asm volatile("cp.async.commit_group;" ::: "memory");
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();   // every warp is done with its tiles: the buffer now holds the merge state
    attn_stamp(tr, 3);
    float* wacc = reinterpret_cast<float*>(asmem);   // [warp][G][HD]
    if (hv) {
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            wacc[(warp * G + gq) * HD + 8 * n + 2 * tq] = o[n][0];
            wacc[(warp * G + gq) * HD + 8 * n + 2 * tq + 1] = o[n][1];
        }
        if (tq == 0) {
            wm[warp][gq] = mrow;
            wl[warp][gq] = lrow;
        }
    }
    __syncthreads();

    const int n_heads = p.n_heads;
    // the cluster form's partial of this split, after the warp-merge state: acc [G][HD], m, l [G]
    float* cacc = wacc + kAttnWarps * G * HD;
    float* cm = cacc + G * HD;
    float* cl = cm + G;
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
            A += wacc[(w * G + h) * HD + d] * f;
        }
        const int hg = g * G + h;
        if (n_active == 1) {
            p.out[((size_t)b * n_heads + hg) * HD + d] = __float2half_rn(A / Ls);
        } else if (CL) {
            cacc[i] = A;
            if (d == 0) {
                cm[h] = M;
                cl[h] = Ls;
            }
        } else {
            const size_t slot = ((size_t)b * n_heads + hg) * p.nsplit + s;
            p.pacc[slot * HD + d] = A;
            if (d == 0) {
                p.pm[slot] = M;
                p.pl[slot] = Ls;
            }
        }
    }
    if (n_active == 1) {
        attn_stamp(tr, 4);
        attn_stamp(tr, 5);
        return;
    }
    if (CL) {
        cluster_barrier();   // every split's partial is in its CTA's shared memory
        attn_stamp(tr, 4);
        // this CTA merges float4 outputs [s * per, s * per + per) of the group's G * HD / 4,
        // over the splits in order (the ticket form's arithmetic and order)
        constexpr int N4 = G * HD / 4, kMergeSplits = 8;
        const int per = (N4 + n_active - 1) / n_active;
        const uint32_t acc_s = static_cast<uint32_t>(__cvta_generic_to_shared(cacc));
        const uint32_t m_s = static_cast<uint32_t>(__cvta_generic_to_shared(cm));
        const uint32_t l_s = static_cast<uint32_t>(__cvta_generic_to_shared(cl));
        for (int j = threadIdx.x; j < per; j += kAttnThreads) {
            const int i = s * per + j;
            if (i >= N4) break;
            const int h = i / (HD / 4), d4 = i - h * (HD / 4);
            float M = -INFINITY, Ls = 0.f;
            float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int k0 = 0; k0 < n_active; k0 += kMergeSplits) {
                float mk[kMergeSplits], lk[kMergeSplits];
                float4 ak[kMergeSplits];
#pragma unroll
                for (int u = 0; u < kMergeSplits; ++u) {
                    if (k0 + u < n_active) {
                        const uint32_t r = (uint32_t)(k0 + u);   // split k is cluster rank k
                        mk[u] = ld_cluster_f32(cluster_addr(m_s + 4u * h, r));
                        lk[u] = ld_cluster_f32(cluster_addr(l_s + 4u * h, r));
                        ak[u] = ld_cluster_f32x4(cluster_addr(acc_s + 16u * (uint32_t)i, r));
                    }
                }
#pragma unroll
                for (int u = 0; u < kMergeSplits; ++u) {
                    if (k0 + u < n_active && mk[u] != -INFINITY) {
                        const float mn = fmaxf(M, mk[u]);
                        const float fo = exp2f(M - mn), fk = exp2f(mk[u] - mn);
                        Ls = Ls * fo + lk[u] * fk;
                        A.x = A.x * fo + ak[u].x * fk; A.y = A.y * fo + ak[u].y * fk;
                        A.z = A.z * fo + ak[u].z * fk; A.w = A.w * fo + ak[u].w * fk;
                        M = mn;
                    }
                }
            }
            const float inv = 1.0f / Ls;
            __half* o = p.out + ((size_t)b * n_heads + g * G + h) * HD + d4 * 4;
            *reinterpret_cast<__half2*>(o) = __floats2half2_rn(A.x * inv, A.y * inv);
            *reinterpret_cast<__half2*>(o + 2) = __floats2half2_rn(A.z * inv, A.w * inv);
        }
        cluster_barrier();   // the other CTAs are done reading this CTA's partial
        if (tr != nullptr && threadIdx.x == 0) tr[6] = 1;
        attn_stamp(tr, 5);
        return;
    }

    // the split ticket: the barrier orders every thread's partial stores before thread 0's
    // release (cumulative), and thread 0's acquire before the merge's loads
    __syncthreads();
    if (threadIdx.x == 0) {
        int ticket;
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(ticket) : "l"(&p.tickets[b * p.n_kv + g]) : "memory");
        last_flag = (ticket == n_active - 1);
    }
    __syncthreads();
    attn_stamp(tr, 4);
    if (!last_flag) {
        attn_stamp(tr, 5);
        return;
    }
    // merge: one pass per float4 output over the splits (online softmax in the exp2 domain),
    // the (m, l, acc) loads of kMergeSplits splits issued together
    for (int i = threadIdx.x; i < G * HD / 4; i += kAttnThreads) {
        const int h = i / (HD / 4), d4 = i - h * (HD / 4);
        const size_t base = ((size_t)b * n_heads + g * G + h) * p.nsplit;
        const float4* srcp = reinterpret_cast<const float4*>(p.pacc) + base * (HD / 4) + d4;
        float M = -INFINITY, Ls = 0.f;
        float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
        constexpr int kMergeSplits = 8;   // 16 raised the kernel to 186 registers (2 CTAs per SM)
        for (int k0 = 0; k0 < n_active; k0 += kMergeSplits) {
            float mk[kMergeSplits], lk[kMergeSplits];
            float4 ak[kMergeSplits];
#pragma unroll
            for (int u = 0; u < kMergeSplits; ++u) {
                if (k0 + u < n_active) {
                    mk[u] = __ldcg(p.pm + base + k0 + u);
                    lk[u] = __ldcg(p.pl + base + k0 + u);
                    ak[u] = __ldcg(srcp + (size_t)(k0 + u) * (HD / 4));
                }
            }
#pragma unroll
            for (int u = 0; u < kMergeSplits; ++u) {
                if (k0 + u < n_active && mk[u] != -INFINITY) {
                    const float mn = fmaxf(M, mk[u]);
                    const float fo = exp2f(M - mn), fk = exp2f(mk[u] - mn);
                    Ls = Ls * fo + lk[u] * fk;
                    A.x = A.x * fo + ak[u].x * fk; A.y = A.y * fo + ak[u].y * fk;
                    A.z = A.z * fo + ak[u].z * fk; A.w = A.w * fo + ak[u].w * fk;
                    M = mn;
                }
            }
        }
        const float inv = 1.0f / Ls;
        __half* o = p.out + ((size_t)b * n_heads + g * G + h) * HD + d4 * 4;
        *reinterpret_cast<__half2*>(o) = __floats2half2_rn(A.x * inv, A.y * inv);
        *reinterpret_cast<__half2*>(o + 2) = __floats2half2_rn(A.z * inv, A.w * inv);
    }
    if (threadIdx.x == 0) p.tickets[b * p.n_kv + g] = 0;   // re-arm for the next call
    if (tr != nullptr && threadIdx.x == 0) tr[6] = 1;   // this CTA merged the splits
    attn_stamp(tr, 5);
}

struct Layout {
    int nsplit, spb;
    size_t tickets_off, pm_off, pl_off, pacc_off, total;
};

Layout layout(int64_t batch, int n_heads, int n_kv, int head_dim, int64_t maxb, int sms) {
    Layout lo = {};
    // Split the block table so that a full-capacity batch gives several CTAs per SM.
    const int64_t pairs = batch * n_kv;
    // about 16 CTAs per SM for a full-capacity batch (mixed context lengths then spread over the
    // SMs evenly; batch 32 over lengths in [128, 8192] measured 5292 tokens/s against 5122 with
    // 8 and 5220 with 32); QL_ATTN_CTAS_PER_SM overrides it for A/B measurements
    static const int env_target = [] {
        const char* e = std::getenv("QL_ATTN_CTAS_PER_SM");
        const int v = e ? std::atoi(e) : 0;
        return v > 0 && v <= 64 ? v : 16;
    }();
    const int64_t target = (int64_t)env_target * sms;
    int64_t spb = (maxb * pairs + target - 1) / target;
    // batch 1-2: two blocks per warp of a CTA, so that a split's blocks are all staged from the
    // start (8 warps, 16 blocks); QL_ATTN_MIN_SPB overrides the floor for A/B measurements
    static const int env_spb = [] {
        const char* e = std::getenv("QL_ATTN_MIN_SPB");
        return e ? std::atoi(e) : 0;
    }();
    // batch 3+: at least 7 blocks per warp, so that a split's pipeline fill and drain stay a
    // small part of it (batch 32 at 2048 positions: 28-block splits 69.5 us, 14-block 79.9 us)
    const int64_t min_spb = env_spb > 0 ? (int64_t)(env_spb > 256 ? 256 : env_spb)
                                        : (batch <= 2 ? 2 * attn_warps(batch) : 7 * attn_warps(batch));
    if (spb < min_spb) spb = min_spb;
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

// Dynamic shared memory of one CTA: the warps' double-buffered K/V tiles, reused afterwards for
// the warp-merge state and the cluster form's split partial.
template <int HD, int G, int NW, bool KQ = false>
constexpr size_t attn_smem() {
    const size_t tile = (size_t)kBS * (HD * 2 + 16);
    const size_t tiles = (size_t)NW * (KQ ? 2 * (size_t)Kvq<HD>::BYTES + 2 * tile : 4 * tile);
    const size_t merge = (size_t)NW * G * HD * 4 + (size_t)G * HD * 4 + 2 * G * 4;
    return tiles > merge ? tiles : merge;
}

constexpr int kMaxCluster = 16;   // splits merged through a cluster (the non-portable maximum)

// Per device: how many clusters of each size (2..16) of the cluster-form kernel can be resident
// at once, by (head_dim 64 | 128, G = 1, 2, 4, 8); filled by attn_prepare.
struct ClusterFit {
    int n[2][4][kMaxCluster + 1];
};
std::mutex g_fit_mu;
std::map<int, ClusterFit> g_fit;
std::atomic<int> g_attn_merge{-1};   // QL_ATTN_MERGE_TICKET / _CLUSTER; -1: from the environment

int attn_merge_form() {
    int f = g_attn_merge.load();
    if (f < 0) {
        const char* e = std::getenv("QL_ATTN_MERGE");
        f = (e != nullptr && std::atoi(e) == QL_ATTN_MERGE_CLUSTER) ? QL_ATTN_MERGE_CLUSTER : QL_ATTN_MERGE_TICKET;
        int expect = -1;
        g_attn_merge.compare_exchange_strong(expect, f);
        f = g_attn_merge.load();
    }
    return f;
}

constexpr int g_index(int G) { return G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3; }

template <int HD, int G>
cudaError_t allow_attn_smem(ClusterFit& fit) {
    cudaError_t e = cudaFuncSetAttribute(attn_split_kernel<HD, G, 4, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)attn_smem<HD, G, 4>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(attn_split_kernel<HD, G, 8, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)attn_smem<HD, G, 8>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(attn_split_kernel<HD, G, 4, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)attn_smem<HD, G, 4, true>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(attn_split_kernel<HD, G, 8, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)attn_smem<HD, G, 8, true>());
    auto* kcl = attn_split_kernel<HD, G, 8, true>;
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kcl, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)attn_smem<HD, G, 8>());
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kcl, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    int* n = fit.n[HD == 64 ? 0 : 1][g_index(G)];
    for (int c = 0; c <= kMaxCluster; ++c) n[c] = 0;
    for (int c = 2; c <= kMaxCluster; ++c) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(c, 1, 1);
        cfg.blockDim = dim3(8 * 32);
        cfg.dynamicSmemBytes = attn_smem<HD, G, 8>();
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = c;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int k = 0;
        if (cudaOccupancyMaxActiveClusters(&k, kcl, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();   // a size the device cannot form: no cluster of it
            k = 0;
        }
        n[c] = k;
    }
    return cudaSuccess;
}

// The cluster form applies at batch 1-2 (8 warps) with 2..16 splits, when every (sequence, kv
// head) of the launch can hold its cluster at the same time.
bool use_cluster(int HD, int G, int nsplit, int n_kv, int batch) {
    if (attn_warps(batch) != 8 || nsplit < 2 || nsplit > kMaxCluster) return false;
    if (attn_merge_form() != QL_ATTN_MERGE_CLUSTER) return false;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lk(g_fit_mu);
    auto it = g_fit.find(dev);
    if (it == g_fit.end()) return false;
    return it->second.n[HD == 64 ? 0 : 1][g_index(G)][nsplit] >= n_kv * batch;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                           bool pdl, unsigned int cx, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cx;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <int HD, int G>
cudaError_t launch_hg(const AParams& p, int batch, cudaStream_t s, bool pdl, DevError* err) {
    dim3 grid(p.nsplit, p.n_kv, batch);
    if (p.kvq != nullptr) {   // quantised pool: the ticket merge
        if (attn_warps(batch) == 8)
            return launch(attn_split_kernel<HD, G, 8, false, true>, grid, dim3(8 * 32), attn_smem<HD, G, 8, true>(), s,
                          pdl, p, err);
        return launch(attn_split_kernel<HD, G, 4, false, true>, grid, dim3(4 * 32), attn_smem<HD, G, 4, true>(), s,
                      pdl, p, err);
    }
    if (use_cluster(HD, G, p.nsplit, p.n_kv, batch))
        return launch_cluster(attn_split_kernel<HD, G, 8, true>, grid, dim3(8 * 32), attn_smem<HD, G, 8>(), s, pdl,
                              (unsigned int)p.nsplit, p, err);
    if (attn_warps(batch) == 8)
        return launch(attn_split_kernel<HD, G, 8, false>, grid, dim3(8 * 32), attn_smem<HD, G, 8>(), s, pdl, p, err);
    return launch(attn_split_kernel<HD, G, 4, false>, grid, dim3(4 * 32), attn_smem<HD, G, 4>(), s, pdl, p, err);
}

template <int HD>
cudaError_t launch_h(const AParams& p, int G, int batch, cudaStream_t s, bool pdl, DevError* err) {
    switch (G) {
        case 1: return launch_hg<HD, 1>(p, batch, s, pdl, err);
        case 2: return launch_hg<HD, 2>(p, batch, s, pdl, err);
        case 4: return launch_hg<HD, 4>(p, batch, s, pdl, err);
        case 8: return launch_hg<HD, 8>(p, batch, s, pdl, err);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

// Kernel attributes (dynamic shared memory above 48 KB) once per device, outside any capture.
int attn_prepare() {
    static std::mutex mu;
    static std::set<int> done;
    int dev = 0;
    QL_TRY_CUDA(cudaGetDevice(&dev));
    std::lock_guard<std::mutex> lk(mu);
    if (done.count(dev)) return QL_OK;
    ClusterFit fit = {};
    cudaError_t e = allow_attn_smem<128, 1>(fit);
    if (e == cudaSuccess) e = allow_attn_smem<128, 2>(fit);
    if (e == cudaSuccess) e = allow_attn_smem<128, 4>(fit);
    if (e == cudaSuccess) e = allow_attn_smem<128, 8>(fit);
    if (e == cudaSuccess) e = allow_attn_smem<64, 1>(fit);
    if (e == cudaSuccess) e = allow_attn_smem<64, 2>(fit);
    if (e == cudaSuccess) e = allow_attn_smem<64, 4>(fit);
    if (e == cudaSuccess) e = allow_attn_smem<64, 8>(fit);
    if (e != cudaSuccess) return cuda_error(e, "attention: cudaFuncSetAttribute");
    {
        std::lock_guard<std::mutex> lf(g_fit_mu);
        g_fit[dev] = fit;
    }
    done.insert(dev);
    return QL_OK;
}

size_t attn_workspace_bytes(int64_t batch, int n_heads, int n_kv_heads, int head_dim,
                            int block_size, int64_t max_blocks_per_seq) {
    (void)block_size;
    if (batch <= 0 || n_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 || max_blocks_per_seq <= 0)
        return 0;
    return layout(batch, n_heads, n_kv_heads, head_dim, max_blocks_per_seq, num_sms()).total;
}

// Alignment the kernel's accesses need: 16-byte cp.async staging of the K/V pools, 32-bit loads
// of q (the non-fused form reads a head row as uint32 pairs) and half2 stores of the output.
// Checked on the host by every entry point, so a misaligned buffer is QL_EINVAL, never a launch.
int attn_check_alignment(const void* q, const void* k_pool, const void* v_pool, const void* out,
                         const char* who) {
    const uintptr_t kv = reinterpret_cast<uintptr_t>(k_pool) | reinterpret_cast<uintptr_t>(v_pool);
    if ((kv & 15) != 0 || (reinterpret_cast<uintptr_t>(out) & 3) != 0 ||
        (reinterpret_cast<uintptr_t>(q) & 3) != 0)
        return set_error(QL_EINVAL, std::string(who) +
                                        ": K/V pools must be 16-byte aligned, q and the output 4-byte aligned");
    return QL_OK;
}

int attn_launch(const AttnArgs& a, cudaStream_t s, bool pdl) {
    QL_REQUIRE((a.q || a.qkv) && ((a.k_pool && a.v_pool) || a.kvq) && a.block_tables && a.out && a.workspace,
               "attention: null pointer");
    QL_REQUIRE(!a.qkv || (a.q_norm && a.k_norm && a.cos_t && a.sin_t && a.positions && a.max_position > 0),
               "attention: the fused qk-norm/RoPE form needs norms, tables and positions");
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
    const void* kpool = a.kvq ? static_cast<const void*>(a.kvq) : static_cast<const void*>(a.k_pool);
    const void* vpool = a.kvq ? static_cast<const void*>(a.kvq) : static_cast<const void*>(a.v_pool);
    if (int rc = attn_check_alignment(a.q, kpool, vpool, a.out, "attention")) return rc;
    if (!device_error_record()) return set_error(QL_ECUDA, "attention: no device error record");
    if (int rc = attn_prepare()) return rc;
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
    p.trace = a.trace;
    p.trace_ctas = a.trace_ctas;
    char* ws = static_cast<char*>(a.workspace);
    p.tickets = reinterpret_cast<int*>(ws + lo.tickets_off);
    p.pm = reinterpret_cast<float*>(ws + lo.pm_off);
    p.pl = reinterpret_cast<float*>(ws + lo.pl_off);
    p.pacc = reinterpret_cast<float*>(ws + lo.pacc_off);
    p.nsplit = lo.nsplit;
    p.spb = lo.spb;
    p.prefetch = a.context_lens == nullptr ? 1 : 0;
    p.next = a.next;
    p.qkv = a.qkv;
    p.q_norm = a.q_norm;
    p.k_norm = a.k_norm;
    p.cos_t = a.cos_t;
    p.sin_t = a.sin_t;
    p.eps = a.eps;
    p.max_position = a.max_position;
    p.kw = const_cast<__half*>(a.k_pool);
    p.vw = const_cast<__half*>(a.v_pool);
    p.kvq = a.kvq;
    cudaError_t e = a.head_dim == 128 ? launch_h<128>(p, G, a.batch, s, pdl, device_error_record())
                                      : launch_h<64>(p, G, a.batch, s, pdl, device_error_record());
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

extern "C" int ql_paged_attn_decode_kvq(const void* d_q, const void* d_pool, const int32_t* d_block_tables,
                                        const int32_t* d_context_lens, int64_t batch, int n_heads, int n_kv_heads,
                                        int head_dim, int block_size, int64_t max_blocks_per_seq, int64_t num_blocks,
                                        float scale, void* d_out, void* d_workspace, size_t workspace_bytes,
                                        void* stream) {
    using namespace ql;
    QL_REQUIRE(d_context_lens && d_pool, "ql_paged_attn_decode_kvq: null pointer");
    AttnArgs a = {};
    a.q = static_cast<const __half*>(d_q);
    a.kvq = static_cast<uint8_t*>(const_cast<void*>(d_pool));
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
    if (batch < 1 || batch > 65535) return set_error(QL_EINVAL, "ql_paged_attn_decode_kvq: batch out of range");
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
    if (int rc = attn_check_alignment(d_q, d_k_pool, d_v_pool, d_out, "ql_paged_attn_decode_noalloc")) return rc;
    const Layout lo = layout(batch, n_heads, n_kv_heads, head_dim, max_blocks_per_seq, num_sms());
    if (lo.total > kNoAllocScratchBytes)
        return set_error(QL_EINVAL, "ql_paged_attn_decode_noalloc: this shape needs " +
                                        std::to_string(lo.total) + " bytes of split-K scratch, more than the " +
                                        std::to_string(kNoAllocScratchBytes) +
                                        " bytes built into the library; use ql_paged_attn_decode with a workspace");
    void* scratch = nullptr;
    if (int rc = noalloc_scratch_address(&scratch)) return rc;
    if (int rc = attn_prepare()) return rc;
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
    const cudaError_t e = head_dim == 128 ? launch_h<128>(p, G, (int)batch, s, true, err)
                                          : launch_h<64>(p, G, (int)batch, s, true, err);
    if (e != cudaSuccess) return cuda_error(e, "ql_paged_attn_decode_noalloc launch");
    return QL_OK;
}

extern "C" int ql_set_attn_merge_form(int form) {
    using namespace ql;
    if (form != QL_ATTN_MERGE_TICKET && form != QL_ATTN_MERGE_CLUSTER)
        return set_error(QL_EINVAL, "ql_set_attn_merge_form: form must be QL_ATTN_MERGE_TICKET or QL_ATTN_MERGE_CLUSTER");
    const int prev = attn_merge_form();
    g_attn_merge.store(form);
    return prev;
}

extern "C" int ql_paged_attn_merge_form(int64_t batch, int n_heads, int n_kv_heads, int head_dim,
                                        int64_t max_blocks_per_seq) {
    using namespace ql;
    if (batch < 1 || batch > 65535 || n_kv_heads <= 0 || n_heads <= 0 || n_heads % n_kv_heads != 0 ||
        (head_dim != 64 && head_dim != 128) || max_blocks_per_seq < 1)
        return set_error(QL_EINVAL, "ql_paged_attn_merge_form: bad shape");
    const int G = n_heads / n_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return set_error(QL_EINVAL, "ql_paged_attn_merge_form: bad GQA group");
    if (int rc = attn_prepare()) return rc;
    const Layout lo = layout(batch, n_heads, n_kv_heads, head_dim, max_blocks_per_seq, num_sms());
    return use_cluster(head_dim, G, lo.nsplit, n_kv_heads, (int)batch) ? QL_ATTN_MERGE_CLUSTER : QL_ATTN_MERGE_TICKET;
}
