// Causal attention of a prefill chunk: the T query tokens of one sequence (positions p0 ..
// p0 + T - 1, their K/V rows already appended) against the sequence's paged K/V cache, reading
// every K/V block once for the whole chunk.
//
// [IL] inferencelayer cuda_llm.rs runs a prompt as sequential decode: token t attends keys
// 0 .. p0 + t. The same result for T tokens at once: per kv head the chunk's T x G query rows
// (G = query heads per kv head) form the MMA's M dimension, so one staged K/V block serves every
// query row; row (t, h) masks the keys past p0 + t. [FK] ferrum-kernels cuda_decode.rs,
// launch_paged_decode_attention: the split over the block table and the merge of the splits'
// (max, sum, acc) partials.
//
// Grid (split, kv head, row group): a CTA of 8 warps takes 128 query rows (warp w: rows 16w ..,
// row r = token r / G, head r % G of the group) and the split's blocks. The CTA stages each block's
// K and V tiles into shared memory (16-byte cp.async, 4 buffers), then every warp computes
// S = Q K^T with mma.sync m16n8k16 (f16 in, f32 out), the online softmax of its 16 rows in the
// exp2 domain, and O += P V (P rounded to f16). The splits' partials are merged by a second kernel.
#include <cuda_fp16.h>
#include <math.h>

#include "ql_chunk_attn.h"
#include "ql_internal.h"

namespace ql {
namespace {

constexpr int kBSk = 16;                  // tokens per K/V block
constexpr int kCW = 8, kCT = kCW * 32;    // warps, threads
constexpr int kRows = kCW * 16;           // query rows per CTA
constexpr int kNS = 4;                    // staged blocks in flight

struct CParams {
    const __half* q;
    const __half* k_pool;
    const __half* v_pool;
    const int32_t* block_table;
    const int32_t* position;
    int T, n_heads, n_kv, G, nsplit, num_blocks, maxb;
    float scale_log2;
    float* pacc;   // [nsplit][T * n_heads][HD]
    float* pm;     // [nsplit][T * n_heads]
    float* pl;
    __half* out;   // [T][n_heads * HD]
};

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The split's blocks of a chunk whose keys end at L (exclusive): nblocks blocks, spb per split.
__device__ __forceinline__ void split_of(int L, int nsplit, int& nblocks, int& spb, int& n_active) {
    nblocks = (L + kBSk - 1) / kBSk;
    spb = (nblocks + nsplit - 1) / nsplit;
    n_active = (nblocks + spb - 1) / spb;
}

template <int HD>
__global__ void __launch_bounds__(kCT) chunk_attn_kernel(CParams p, DevError* err) {
    constexpr int KSTEPS = HD / 16, NT = HD / 8;
    constexpr int PITCH = HD * 2 + 16;            // bytes per staged row (ldmatrix without bank conflicts)
    constexpr int TILE = kBSk * PITCH;
    constexpr int CHUNKS = HD * 2 / 16;           // 16-byte chunks per row
    extern __shared__ __align__(16) unsigned char csm[];   // [kNS][K | V] tiles
    const int s = blockIdx.x, g = blockIdx.y, z = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, tq = lane & 3;
    pdl_wait();
    pdl_trigger();
    const int p0 = *p.position;
    const int L = p0 + p.T;
    int nblocks, spb, n_active;
    split_of(L, p.nsplit, nblocks, spb, n_active);
    if (s >= n_active) return;
    const int blk0 = s * spb, blk1 = min(nblocks, blk0 + spb);
    const int R = p.T * p.G;                      // query rows of this kv head
    const int r0 = z * kRows + warp * 16;         // this warp's first row
    const int ra = r0 + gq, rb = ra + 8;          // this lane's rows
    const bool va = ra < R, vb = rb < R;
    const int posa = p0 + (va ? ra / p.G : 0), posb = p0 + (vb ? rb / p.G : 0);
    const int heada = g * p.G + (va ? ra % p.G : 0), headb = g * p.G + (vb ? rb % p.G : 0);
    const bool warp_live = r0 < R;
    // the CTA's last query position: blocks after it are masked for every row
    const int rlast = min(R, z * kRows + kRows) - 1;
    const int pos_max = p0 + rlast / p.G;
    const int blk_end = min(blk1, pos_max / kBSk + 1);

    // Q fragments (rows ra, rb of the A operand), k-step kk: dims 16 kk + 2 tq (+8)
    uint32_t qa[KSTEPS][4];
    {
        const uint32_t* qra = reinterpret_cast<const uint32_t*>(p.q + ((size_t)(posa - p0) * p.n_heads + heada) * HD);
        const uint32_t* qrb = reinterpret_cast<const uint32_t*>(p.q + ((size_t)(posb - p0) * p.n_heads + headb) * HD);
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk) {
            qa[kk][0] = va ? qra[8 * kk + tq] : 0u;
            qa[kk][1] = vb ? qrb[8 * kk + tq] : 0u;
            qa[kk][2] = va ? qra[8 * kk + 4 + tq] : 0u;
            qa[kk][3] = vb ? qrb[8 * kk + 4 + tq] : 0u;
        }
    }
    const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(csm));
    // stage block blk into buffer b (every thread a share of the 16-byte copies); a bad block
    // id is recorded and its tiles left as they are (the keys are then masked)
    auto stage = [&](int blk, int b) -> bool {
        const int phys = blk < p.maxb ? __ldg(p.block_table + blk) : -1;   // past the table: invalid
        const bool ok = phys >= 0 && phys < p.num_blocks;
        if (ok) {
            const __half* ks = p.k_pool + ((size_t)phys * p.n_kv + g) * kBSk * HD;
            const __half* vs = p.v_pool + ((size_t)phys * p.n_kv + g) * kBSk * HD;
            const uint32_t kd = sbase + (uint32_t)(b * 2 * TILE), vd = kd + TILE;
            for (int c = tid; c < kBSk * CHUNKS; c += kCT) {
                const int row = c / CHUNKS, col = c - row * CHUNKS;
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(kd + row * PITCH + col * 16),
                             "l"(ks + row * HD + col * 8) : "memory");
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(vd + row * PITCH + col * 16),
                             "l"(vs + row * HD + col * 8) : "memory");
            }
        } else if (tid == 0) {
            record_device_error(err, kErrAttnBlock, blk, phys);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        return ok;
    };
    unsigned okm = 0u;   // bit b: buffer b holds a valid block
    const int nb = blk_end > blk0 ? blk_end - blk0 : 0;
#pragma unroll
    for (int j = 0; j < kNS - 1; ++j) {
        if (j < nb) okm |= (stage(blk0 + j, j) ? 1u : 0u) << j;
        else asm volatile("cp.async.commit_group;" ::: "memory");
    }

    float o[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float ma = -INFINITY, mb_ = -INFINITY, la = 0.f, lb = 0.f;
    const int lm = lane >> 3, lr = lane & 7;
    for (int i = 0; i < nb; ++i) {
        // groups committed: blocks 0 .. i + kNS - 2; block i has landed when at most kNS - 2 pend
        asm volatile("cp.async.wait_group %0;" ::"n"(kNS - 2) : "memory");
        __syncthreads();
        const int blk = blk0 + i, b = i % kNS;
        if (warp_live && ((okm >> b) & 1u)) {
            const uint32_t ksm = sbase + (uint32_t)(b * 2 * TILE), vsm = ksm + TILE;
            // ---- S = Q K^T for the block's 16 keys
            float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
                uint32_t b0, b1, b2, b3;
                const uint32_t addr = ksm + (uint32_t)(((lm >> 1) * 8 + lr) * PITCH + (16 * kk + (lm & 1) * 8) * 2);
                asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                             : "=r"(b0), "=r"(b1), "=r"(b2), "=r"(b3) : "r"(addr));
                mma16816(s0, qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
                mma16816(s1, qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
            }
            // ---- causal mask and online softmax of rows ra (s*[0..1]) and rb (s*[2..3])
            const int k0 = blk * kBSk + 2 * tq;
            const float xa0 = va && k0 <= posa ? s0[0] * p.scale_log2 : -INFINITY;
            const float xa1 = va && k0 + 1 <= posa ? s0[1] * p.scale_log2 : -INFINITY;
            const float xa2 = va && k0 + 8 <= posa ? s1[0] * p.scale_log2 : -INFINITY;
            const float xa3 = va && k0 + 9 <= posa ? s1[1] * p.scale_log2 : -INFINITY;
            const float xb0 = vb && k0 <= posb ? s0[2] * p.scale_log2 : -INFINITY;
            const float xb1 = vb && k0 + 1 <= posb ? s0[3] * p.scale_log2 : -INFINITY;
            const float xb2 = vb && k0 + 8 <= posb ? s1[2] * p.scale_log2 : -INFINITY;
            const float xb3 = vb && k0 + 9 <= posb ? s1[3] * p.scale_log2 : -INFINITY;
            float mxa = fmaxf(fmaxf(xa0, xa1), fmaxf(xa2, xa3));
            float mxb = fmaxf(fmaxf(xb0, xb1), fmaxf(xb2, xb3));
            mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 1));
            mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 2));
            mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 1));
            mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 2));
            const float mna = fmaxf(ma, mxa), mnb = fmaxf(mb_, mxb);
            // a row with no key so far keeps its zero sums (reference 0 instead of -inf)
            const float ra_ = mna == -INFINITY ? 0.f : mna, rb_ = mnb == -INFINITY ? 0.f : mnb;
            const float aa = exp2f(ma - ra_), ab = exp2f(mb_ - rb_);
            const float pa0 = exp2f(xa0 - ra_), pa1 = exp2f(xa1 - ra_), pa2 = exp2f(xa2 - ra_), pa3 = exp2f(xa3 - ra_);
            const float pb0 = exp2f(xb0 - rb_), pb1 = exp2f(xb1 - rb_), pb2 = exp2f(xb2 - rb_), pb3 = exp2f(xb3 - rb_);
            float sa = (pa0 + pa1) + (pa2 + pa3), sb = (pb0 + pb1) + (pb2 + pb3);
            sa += __shfl_xor_sync(0xffffffffu, sa, 1);
            sa += __shfl_xor_sync(0xffffffffu, sa, 2);
            sb += __shfl_xor_sync(0xffffffffu, sb, 1);
            sb += __shfl_xor_sync(0xffffffffu, sb, 2);
            la = la * aa + sa;
            lb = lb * ab + sb;
            ma = mna;
            mb_ = mnb;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                o[n][0] *= aa;
                o[n][1] *= aa;
                o[n][2] *= ab;
                o[n][3] *= ab;
            }
            const __half2 h0 = __floats2half2_rn(pa0, pa1), h1 = __floats2half2_rn(pb0, pb1);
            const __half2 h2 = __floats2half2_rn(pa2, pa3), h3 = __floats2half2_rn(pb2, pb3);
            const uint32_t u0 = *reinterpret_cast<const uint32_t*>(&h0), u1 = *reinterpret_cast<const uint32_t*>(&h1);
            const uint32_t u2 = *reinterpret_cast<const uint32_t*>(&h2), u3 = *reinterpret_cast<const uint32_t*>(&h3);
            // ---- O += P V (V^T fragments by transposing ldmatrix)
#pragma unroll
            for (int pp = 0; pp < NT / 2; ++pp) {
                uint32_t v0, v1, v2, v3;
                const uint32_t addr = vsm + (uint32_t)(((lm & 1) * 8 + lr) * PITCH + (16 * pp + (lm >> 1) * 8) * 2);
                asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                             : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3) : "r"(addr));
                mma16816(o[2 * pp], u0, u1, u2, u3, v0, v1);
                mma16816(o[2 * pp + 1], u0, u1, u2, u3, v2, v3);
            }
        }
        __syncthreads();   // every warp is done with buffer b
        if (i + kNS - 1 < nb) {
            const int nbuf = (i + kNS - 1) % kNS;
            okm = (okm & ~(1u << nbuf)) | ((stage(blk0 + i + kNS - 1, nbuf) ? 1u : 0u) << nbuf);
        } else {
            asm volatile("cp.async.commit_group;" ::: "memory");
        }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    // this split's partial of rows ra, rb: sums, max and the unnormalised output
    const int NR = p.T * p.n_heads;
    const size_t rowa = (size_t)(posa - p0) * p.n_heads + heada, rowb = (size_t)(posb - p0) * p.n_heads + headb;
    if (va) {
#pragma unroll
        for (int n = 0; n < NT; ++n)
            *reinterpret_cast<float2*>(p.pacc + ((size_t)s * NR + rowa) * HD + 8 * n + 2 * tq) = make_float2(o[n][0], o[n][1]);
        if (tq == 0) {
            p.pm[(size_t)s * NR + rowa] = ma;
            p.pl[(size_t)s * NR + rowa] = la;
        }
    }
    if (vb) {
#pragma unroll
        for (int n = 0; n < NT; ++n)
            *reinterpret_cast<float2*>(p.pacc + ((size_t)s * NR + rowb) * HD + 8 * n + 2 * tq) = make_float2(o[n][2], o[n][3]);
        if (tq == 0) {
            p.pm[(size_t)s * NR + rowb] = mb_;
            p.pl[(size_t)s * NR + rowb] = lb;
        }
    }
}

// out[row] = sum_s acc_s 2^(m_s - M) / sum_s l_s 2^(m_s - M), M = max_s m_s, over the active
// splits in order; one warp per (token, head) row. Lane s reads split s's max and sum (one round
// of loads for up to 32 splits), the warp reduces them; then lane = 4 output dims, the splits'
// accumulators loaded 8 at a time (the first 8 together with the max and sum) and added in split
// order.
template <int HD>
__global__ void __launch_bounds__(256) chunk_merge_kernel(CParams p) {
    pdl_wait();
    pdl_trigger();
    const int p0 = *p.position;
    int nblocks, spb, n_active;
    split_of(p0 + p.T, p.nsplit, nblocks, spb, n_active);
    const int NR = p.T * p.n_heads;
    const int lane = threadIdx.x & 31;
    for (int row = blockIdx.x * 8 + (threadIdx.x >> 5); row < NR; row += gridDim.x * 8) {
        // the first 32 splits' (m, l) are loaded once (a chunk rarely has more splits), together
        // with the first round of partial sums, which do not depend on the maximum
        constexpr int kRound = 8;   // partial sums whose loads are in flight together
        const float m0 = lane < n_active ? __ldcg(p.pm + (size_t)lane * NR + row) : -INFINITY;
        const float l0 = lane < n_active ? __ldcg(p.pl + (size_t)lane * NR + row) : 0.f;
        float4 a[kRound];
#pragma unroll
        for (int u = 0; u < kRound; ++u)
            if (u < n_active && lane < HD / 4)
                a[u] = __ldcg(reinterpret_cast<const float4*>(p.pacc + ((size_t)u * NR + row) * HD) + lane);
        float M = -INFINITY;
        for (int s0 = 0; s0 < n_active; s0 += 32) {   // max over the splits
            const int s = s0 + lane;
            const float ms = s0 == 0 ? m0 : s < n_active ? __ldcg(p.pm + (size_t)s * NR + row) : -INFINITY;
            float m = ms;
#pragma unroll
            for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            M = fmaxf(M, m);
        }
        float Ls = 0.f;
        float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s0 = 0; s0 < n_active; s0 += 32) {
            const int ns = n_active - s0 < 32 ? n_active - s0 : 32;
            // lane s: split s0 + s's weight 2^(m - M) and weighted sum
            const int sl = s0 + lane;
            const float ms = s0 == 0 ? m0 : lane < ns ? __ldcg(p.pm + (size_t)sl * NR + row) : -INFINITY;
            const float ls = s0 == 0 ? l0 : lane < ns ? __ldcg(p.pl + (size_t)sl * NR + row) : 0.f;
            const float f = ms == -INFINITY ? 0.f : exp2f(ms - M);
            // the splits' sums in split order (lane 0 adds them after a gather)
            float lw = ls * f;
            for (int k = 0; k < ns; ++k) Ls += __shfl_sync(0xffffffffu, lw, k);
            for (int k0 = 0; k0 < ns; k0 += kRound) {
                float fk[kRound];
#pragma unroll
                for (int u = 0; u < kRound; ++u) {
                    fk[u] = __shfl_sync(0xffffffffu, f, (k0 + u) & 31);
                    // the first round's loads went out with the (m, l) above
                    if ((s0 > 0 || k0 > 0) && k0 + u < ns && lane < HD / 4)
                        a[u] = __ldcg(reinterpret_cast<const float4*>(p.pacc + ((size_t)(s0 + k0 + u) * NR + row) * HD) + lane);
                }
#pragma unroll
                for (int u = 0; u < kRound; ++u) {
                    if (k0 + u < ns && lane < HD / 4) {
                        A.x = fmaf(a[u].x, fk[u], A.x);
                        A.y = fmaf(a[u].y, fk[u], A.y);
                        A.z = fmaf(a[u].z, fk[u], A.z);
                        A.w = fmaf(a[u].w, fk[u], A.w);
                    }
                }
            }
        }
        if (lane < HD / 4) {
            const float inv = 1.0f / Ls;
            __half2* dst = reinterpret_cast<__half2*>(p.out + (size_t)row * HD) + 2 * lane;
            dst[0] = __floats2half2_rn(A.x * inv, A.y * inv);
            dst[1] = __floats2half2_rn(A.z * inv, A.w * inv);
        }
    }
}

template <int HD>
constexpr size_t chunk_smem() {
    return (size_t)kNS * 2 * kBSk * (HD * 2 + 16);
}

int chunk_nsplit(int n_kv, int T, int G) {
    const int nz = (T * G + kRows - 1) / kRows;
    int ns = (num_sms() + n_kv * nz - 1) / (n_kv * nz);
    return ns < 1 ? 1 : (ns > 64 ? 64 : ns);
}

}  // namespace

size_t chunk_attn_workspace_bytes(int T, int n_heads, int n_kv, int head_dim) {
    if (T < 1 || n_kv < 1 || n_heads % n_kv) return 0;
    const size_t ns = (size_t)chunk_nsplit(n_kv, T, n_heads / n_kv);
    const size_t rows = (size_t)T * n_heads;
    return ns * rows * ((size_t)head_dim + 2) * sizeof(float) + 256;
}

int chunk_attn_launch(const ChunkAttnArgs& a, cudaStream_t st, bool pdl) {
    QL_REQUIRE(a.q && a.k_pool && a.v_pool && a.block_table && a.position && a.out && a.workspace,
               "chunk attention: null pointer");
    QL_REQUIRE(a.head_dim == 64 || a.head_dim == 128, "chunk attention: head_dim must be 64 or 128");
    QL_REQUIRE(a.n_kv_heads > 0 && a.n_heads % a.n_kv_heads == 0, "chunk attention: n_heads % n_kv_heads != 0");
    QL_REQUIRE(a.T >= 1 && a.T <= 256, "chunk attention: 1..256 tokens");
    QL_REQUIRE(a.workspace_bytes >= chunk_attn_workspace_bytes(a.T, a.n_heads, a.n_kv_heads, a.head_dim),
               "chunk attention: workspace too small");
    DevError* err = device_error_record();
    if (!err) return set_error(QL_ECUDA, "chunk attention: no device error record");
    const int G = a.n_heads / a.n_kv_heads;
    const int nz = (a.T * G + kRows - 1) / kRows;
    CParams p = {};
    p.q = a.q;
    p.k_pool = a.k_pool;
    p.v_pool = a.v_pool;
    p.block_table = a.block_table;
    p.position = a.position;
    p.T = a.T;
    p.n_heads = a.n_heads;
    p.n_kv = a.n_kv_heads;
    p.G = G;
    p.nsplit = chunk_nsplit(a.n_kv_heads, a.T, G);
    p.num_blocks = a.num_blocks;
    p.maxb = a.max_blocks_per_seq;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    const size_t rows = (size_t)a.T * a.n_heads;
    p.pacc = static_cast<float*>(a.workspace);
    p.pm = p.pacc + (size_t)p.nsplit * rows * a.head_dim;
    p.pl = p.pm + (size_t)p.nsplit * rows;
    p.out = a.out;
    const dim3 grid(p.nsplit, a.n_kv_heads, nz);
    cudaError_t e;
    static_assert(chunk_smem<128>() <= 48 * 1024, "the staged tiles fit the default shared-memory limit");
    if (a.head_dim == 128) {
        e = launch(chunk_attn_kernel<128>, grid, dim3(kCT), chunk_smem<128>(), st, pdl, p, err);
        if (e == cudaSuccess)
            e = launch(chunk_merge_kernel<128>, dim3(2 * num_sms()), dim3(256), 0, st, pdl, p);
    } else {
        e = launch(chunk_attn_kernel<64>, grid, dim3(kCT), chunk_smem<64>(), st, pdl, p, err);
        if (e == cudaSuccess)
            e = launch(chunk_merge_kernel<64>, dim3(2 * num_sms()), dim3(256), 0, st, pdl, p);
    }
    return e == cudaSuccess ? QL_OK : cuda_error(e, "chunk attention launch");
}

}  // namespace ql

extern "C" size_t ql_paged_attn_chunk_workspace_bytes(int64_t n_tokens, int n_heads, int n_kv_heads, int head_dim) {
    if (n_tokens < 1 || n_tokens > 256 || (head_dim != 64 && head_dim != 128)) return 0;
    return ql::chunk_attn_workspace_bytes((int)n_tokens, n_heads, n_kv_heads, head_dim);
}

extern "C" int ql_paged_attn_chunk(const void* d_q, const void* d_k_pool, const void* d_v_pool,
                                   const int32_t* d_block_table, const int32_t* d_position, int64_t n_tokens,
                                   int n_heads, int n_kv_heads, int head_dim, int block_size,
                                   int64_t max_blocks_per_seq, int64_t num_blocks, float scale, void* d_out,
                                   void* d_workspace, size_t workspace_bytes, void* stream) {
    using namespace ql;
    QL_REQUIRE(block_size == 16, "ql_paged_attn_chunk: block_size must be 16");
    QL_REQUIRE(max_blocks_per_seq >= 1 && max_blocks_per_seq < (1ll << 26) && num_blocks >= 1 &&
                   num_blocks < (1ll << 31),
               "ql_paged_attn_chunk: bad table or pool size");
    QL_REQUIRE(n_tokens >= 1 && n_tokens <= 256, "ql_paged_attn_chunk: 1..256 tokens");
    QL_REQUIRE((reinterpret_cast<uintptr_t>(d_k_pool) & 15) == 0 && (reinterpret_cast<uintptr_t>(d_v_pool) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(d_q) & 3) == 0 && (reinterpret_cast<uintptr_t>(d_out) & 3) == 0,
               "ql_paged_attn_chunk: K/V pools must be 16-byte aligned, q and the output 4-byte aligned");
    ChunkAttnArgs a = {};
    a.q = static_cast<const __half*>(d_q);
    a.k_pool = static_cast<const __half*>(d_k_pool);
    a.v_pool = static_cast<const __half*>(d_v_pool);
    a.block_table = d_block_table;
    a.position = d_position;
    a.T = (int)n_tokens;
    a.n_heads = n_heads;
    a.n_kv_heads = n_kv_heads;
    a.head_dim = head_dim;
    a.max_blocks_per_seq = (int)max_blocks_per_seq;
    a.num_blocks = (int)num_blocks;
    a.scale = scale;
    a.out = static_cast<__half*>(d_out);
    a.workspace = d_workspace;
    a.workspace_bytes = workspace_bytes;
    return chunk_attn_launch(a, static_cast<cudaStream_t>(stream), false);
}
