// Model handle and the whole decode step.
//
// [IL] inferencelayer cuda_llm.rs CudaQwen3::step / seed / capture / run_graph: a step takes
// no host arguments (token, position and KV offset live in device memory), allocates
// nothing, and is captured once as a CUDA graph that every later step replays; greedy argmax
// and the position advance stay on the device. [FK] ferrum-kernels cuda_decode.rs
// batch_decode_step: several sequences per step over a paged KV pool.
//
// With QL_OPT_STEP_KERNEL = QL_STEP_PERSISTENT (batches up to ql_model_persistent_max_batch())
// the step runs as ONE cooperative kernel (ql_persist.cuh). Otherwise (the default) it runs
// this kernel sequence, all launched with programmatic dependent launch so that each GEMV
// starts streaming its weights while its predecessor drains; at batch 1-2 the GEMVs read the
// tile stream copy of the weights (stream_gemv_launch), above that the row-major q4_0 arrays:
//   embed                      x[b] = E[token[b]]                          (f32 residual)
//   per layer:
//     gemv  rms(x)*attn_norm -> W_qkv                                       -> qkv f32
//     norm_rope                q/k RMSNorm + RoPE, K/V -> paged pool        -> q f16
//     attention                split-K paged GQA over positions 0..p       -> o f16
//     gemv  o -> W_o, x += .                                                (residual epilogue)
//     gemv  rms(x)*ffn_norm -> W_gate|up, silu(g)*u                         -> act f16
//     gemv  act -> W_down, x += .                                           (residual epilogue)
//   gemv  rms(x)*final_norm -> W_lm, logits + packed argmax keys
//   finalize                   next token, position += 1, keys re-armed
#include <cuda_fp16.h>

#include <cstdlib>
#include <map>
#include <vector>

#include "ql_batched.h"
#include "ql_chunk_attn.h"
#include "ql_internal.h"

struct ql_model {
    ql_model_desc d;
    std::vector<ql_layer_desc> layers;
    int device = 0;
    // workspace (owned)
    float* x = nullptr;          // [maxB][hidden]
    float* qkv = nullptr;        // [maxB][qkv_rows]
    __half* q16 = nullptr;       // [maxB][nh*hd]
    __half* attn = nullptr;      // [maxB][nh*hd]
    __half* act = nullptr;       // [maxB][inter]
    float* logits = nullptr;     // [maxB][vocab]
    unsigned long long* keys = nullptr;   // [maxB]
    float* cos_t = nullptr;      // [max_pos][hd/2]
    float* sin_t = nullptr;
    void* attn_ws = nullptr;
    size_t attn_ws_bytes = 0;
    std::vector<void*> owned;
    std::map<int64_t, cudaGraphExec_t> graphs;
    std::map<int64_t, ql_step_args> graph_args;   // the device buffers each graph was captured with
    // L2 prefetch of the following GEMV's weights by every kernel (A/B switch QL_NEXT_PREFETCH=1).
    // Off by default: measured slower (kernels that issue megabytes of prefetch stall).
    bool next_prefetch = false;
    // persistent step kernel (one cooperative launch per step) for batches up to persist_max_b
    int persist_max_b = 0;                  // 0: not available for this shape / device
    int step_kernel = QL_STEP_AUTO;
    unsigned long long barrier_timeout_ns = 2000000000ull;
    unsigned int barrier_extra = 0;
    unsigned long long* trace = nullptr;    // caller-owned, see QL_OPT_STEP_TRACE
    unsigned long long* mtrace = nullptr;   // caller-owned, see QL_OPT_MERGE_TRACE
    ql::PLayer* players = nullptr;          // device [n_layers]
    uint8_t* pstreams = nullptr;            // all matrices in the tile stream layout
    size_t persist_stream_bytes = 0;
    std::vector<ql::PMat> hmats;            // host copies: 4 per layer, then lm_head
    unsigned int* ssync = nullptr;          // abort flag of the stand-alone stream GEMVs
    float* ssq = nullptr;                   // batch 3-32: 32-row chunk sums of x^2 ([hidden / 32][32])
    __half* xn = nullptr;                   // [max_batch][hidden] RMSNorm'd input of a batched GEMV
    void* bws = nullptr;                    // batched GEMV partial sums
    size_t bws_bytes = 0;
    bool batched_ok = false;                // every matrix width suits the batched stream GEMV
    ql::PMat plm = {};
    int max_nblk = 0, persist_nsplit = 1;
    float* ppm = nullptr;
    float* ppl = nullptr;
    float* ppacc = nullptr;
    int* ptickets = nullptr;
    unsigned int* psync = nullptr;
    // routed experts (num_experts > 0): the router's logits and ticket, the selection, the
    // selected experts' SiLU*up activations and down outputs
    float* mlog = nullptr;       // [num_experts]
    int* mticket = nullptr;
    int32_t* meidx = nullptr;    // [topk]
    float* mewt = nullptr;       // [topk]
    __half* mact = nullptr;      // [topk][moe_inter]
    float* medn = nullptr;       // [topk][hidden]
    // chunked prefill: the chunk's per-token block tables (the sequence's row repeated),
    // positions and context lengths
    int32_t* pbt = nullptr;      // [max_batch][max_blocks_per_seq]
    int32_t* ppos = nullptr;     // [max_batch]
    int32_t* plen = nullptr;     // [max_batch]
    void* cws = nullptr;         // prefill chunk attention: the splits' partials
    size_t cws_bytes = 0;
    void* gws = nullptr;         // prefill GEMM: the K parts' sums of matrices with few row blocks
    size_t gws_bytes = 0;
};

namespace ql {
namespace {

__global__ void embed_kernel(const float* __restrict__ E, const int32_t* __restrict__ tokens,
                             const int32_t* __restrict__ active, float* __restrict__ x, int hidden,
                             int vocab, DevError* err, NextWeights next) {
    const int b = blockIdx.x;
    l2_prefetch_share(next.ptr[0], next.bytes[0]);
    l2_prefetch_share(next.ptr[1], next.bytes[1]);
    pdl_wait();
    pdl_trigger();
    int tok = tokens[b];
    const bool act = active == nullptr || active[b] != 0;
    if (tok < 0 || tok >= vocab) {
        if (act && threadIdx.x == 0) record_device_error(err, kErrEmbedToken, b, tok);
        tok = 0;
    }
    const float4* src = reinterpret_cast<const float4*>(E + (size_t)tok * hidden);
    float4* dst = reinterpret_cast<float4*>(x + (size_t)b * hidden);
    for (int i = threadIdx.x; i < hidden / 4; i += blockDim.x) dst[i] = src[i];
}

__global__ void finalize_kernel(unsigned long long* keys, const int32_t* active, int32_t* positions,
                                int32_t* next_tokens, int32_t* out_tokens, long long out_stride,
                                float* logits_dummy, int batch) {
    (void)logits_dummy;
    pdl_wait();
    pdl_trigger();
    for (int b = threadIdx.x; b < batch; b += blockDim.x) {
        const unsigned long long k = keys[b];
        keys[b] = 0ull;
        if (active && active[b] == 0) continue;
        const int tok = (int)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull));
        const int pos = positions[b];
        next_tokens[b] = tok;
        if (out_tokens && pos + 1 >= 0 && pos + 1 < out_stride)
            out_tokens[(size_t)b * out_stride + pos + 1] = tok;
        positions[b] = pos + 1;
    }
}

// Chunked prefill: token t of the chunk sits at position p0 + t (p0 = *position) and attends
// to positions 0 .. p0 + t; every token uses the sequence's block table row.
__global__ void prefill_setup_kernel(const int32_t* position, const int32_t* block_table, int maxb, int T,
                                     int32_t* bt, int32_t* pos, int32_t* len) {
    pdl_wait();
    pdl_trigger();
    const int p0 = *position;
    for (int i = threadIdx.x; i < T * maxb; i += blockDim.x) bt[i] = block_table[i % maxb];
    for (int t = threadIdx.x; t < T; t += blockDim.x) {
        pos[t] = p0 + t;
        len[t] = p0 + t + 1;
    }
}

// The chunk's last token's greedy next token (its argmax key), the position advanced by T.
__global__ void prefill_finish_kernel(unsigned long long* keys, int32_t* position, int32_t* next_token, int T) {
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x != 0) return;
    const unsigned long long k = keys[0];
    keys[0] = 0ull;
    if (next_token) *next_token = (int)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull));
    *position += T;
}

bool check_matrix(const ql_q4_0_matrix& m, int64_t rows, int64_t cols) {
    return m.scales && m.quants && m.rows == rows && m.cols == cols;
}

int alloc(ql_model* m, void** p, size_t bytes) {
    cudaError_t e = cudaMalloc(p, bytes);
    if (e != cudaSuccess) return set_error(QL_ENOMEM, std::string("ql_model_create: cudaMalloc failed: ") + cudaGetErrorString(e));
    m->owned.push_back(*p);
    return QL_OK;
}

// CTAs of the o GEMV at batch 1-2: the SMs minus the attention's merging CTAs (they end last),
// if that keeps the largest per-CTA tile count; else one per SM (0). QL_O_GEMV_FULL=1 keeps
// one per SM for A/B measurements.
int o_gemv_grid(int sms, int mergers, int ntile) {
    static const bool full = [] {
        const char* e = std::getenv("QL_O_GEMV_FULL");
        return e != nullptr && std::atoi(e) != 0;
    }();
    const int g = sms - mergers;
    if (full || g <= 0 || g >= sms) return 0;
    const int per_full = (ntile + sms - 1) / sms, per_less = (ntile + g - 1) / g;
    return per_less == per_full ? g : 0;
}

// The whole step as one cooperative kernel (ql_persist.cuh).
int run_persist(ql_model* m, const ql_step_args* a, cudaStream_t s) {
    const ql_model_desc& d = m->d;
    const int B = (int)a->batch;
    PersistParams p = {};
    p.layers = m->players;
    p.n_layers = (int)d.n_layers;
    p.lm = m->plm;
    p.final_norm = d.final_norm;
    p.embed = d.embed;
    p.hidden = (int)d.hidden;
    p.inter = (int)d.intermediate;
    p.vocab = (int)d.vocab;
    p.nh = (int)d.n_heads;
    p.nkv = (int)d.n_kv_heads;
    p.B = B;
    p.maxb = (int)d.max_blocks_per_seq;
    int nsplit = num_sms() / (B * (int)d.n_kv_heads);
    nsplit = nsplit < 1 ? 1 : nsplit > m->persist_nsplit ? m->persist_nsplit : nsplit;
    p.nsplit = nsplit;
    p.max_nblk = m->max_nblk;
    p.eps = d.eps;
    p.scale_log2 = 1.4426950408889634f / sqrtf((float)d.head_dim);
    p.num_blocks = d.num_blocks;
    p.layer_pool = (long long)d.num_blocks * d.n_kv_heads * d.block_size * d.head_dim;
    p.max_position = d.max_blocks_per_seq * d.block_size;
    p.out_stride = a->out_tokens ? a->out_stride : 0;
    p.barrier_timeout_ns = m->barrier_timeout_ns;
    p.barrier_extra = m->barrier_extra;
    p.trace = m->trace;
    p.tokens = a->tokens;
    p.positions = a->positions;
    p.block_tables = a->block_tables;
    p.active = a->active;
    p.next_tokens = a->next_tokens;
    p.out_tokens = a->out_tokens;
    p.logits = a->logits ? a->logits : m->logits;
    p.x = m->x;
    p.qkv = m->qkv;
    p.attn = m->attn;
    p.act = m->act;
    p.keys = m->keys;
    p.cos_t = m->cos_t;
    p.sin_t = m->sin_t;
    p.k_pool = static_cast<__half*>(d.k_pool);
    p.v_pool = static_cast<__half*>(d.v_pool);
    p.pm = m->ppm;
    p.pl = m->ppl;
    p.pacc = m->ppacc;
    p.tickets = m->ptickets;
    p.sync = m->psync;
    p.err = device_error_record();
    if (!p.err) return set_error(QL_ECUDA, "decode step: no device error record");
    return persist_launch(p, (int)d.head_dim, (int)(d.n_heads / d.n_kv_heads), s);
}

int run_step(ql_model* m, const ql_step_args* a, cudaStream_t s) {
    const ql_model_desc& d = m->d;
    const int B = (int)a->batch;
    if (m->step_kernel == QL_STEP_PERSISTENT && B > m->persist_max_b)
        return set_error(QL_EINVAL, "decode step: the persistent step kernel takes batches up to " +
                                        std::to_string(m->persist_max_b) + " on this model");
    if (m->step_kernel == QL_STEP_PERSISTENT && (m->d.kv_format != QL_KV_F16 || m->d.num_experts > 0))
        return set_error(QL_EINVAL, "decode step: the persistent step kernel takes only dense models with f16 KV");
    if (m->d.num_experts > 0 && B != 1)
        return set_error(QL_EINVAL, "decode step: routed experts decode at batch 1");
    if (m->d.num_experts > 0 && m->hmats.empty())
        return set_error(QL_EINVAL, "decode step: routed experts need the tile stream copies (matrix widths multiples of 128)");
    if (m->step_kernel == QL_STEP_PERSISTENT) return run_persist(m, a, s);
    const bool pdl = true;
    const int hd = (int)d.head_dim, nh = (int)d.n_heads, nkv = (int)d.n_kv_heads;
    const size_t layer_pool = (size_t)d.num_blocks * nkv * d.block_size * hd;
    const bool kvq = d.kv_format == QL_KV_Q8_0_Q5_1;
    const size_t kvq_layer = (size_t)d.num_blocks * nkv * (size_t)ql_kvq_record_bytes(hd);
    int rc;

    // Each kernel asks L2 to fetch the weights of a GEMV that follows it, so that HBM keeps
    // streaming weights through kernel boundaries, launches and the small kernels:
    //   embed -> qkv(0); qkv(l) -> o(l); norm_rope(l) -> gate|up(l); gate|up(l) -> down(l);
    //   down(l) -> qkv(l+1), or the first 64 MB of lm_head after the last layer.
    const bool pf = m->next_prefetch;
    auto nw = [pf](const ql_q4_0_matrix& w, size_t cap) {
        NextWeights n = {};
        if (!pf) return n;
        const size_t qb = (size_t)w.rows * w.cols / 2, sb = (size_t)w.rows * w.cols / 16;
        n.ptr[0] = w.quants;
        n.bytes[0] = qb < cap ? qb : cap;
        n.ptr[1] = w.scales;
        n.bytes[1] = sb < cap / 8 ? sb : cap / 8;
        return n;
    };
    const size_t kAll = ~(size_t)0, kLmHead = (size_t)64 << 20;
    cudaError_t e = launch(embed_kernel, dim3(B), dim3(256), 0, s, pdl, d.embed, a->tokens, a->active,
                           m->x, (int)d.hidden, (int)d.vocab, device_error_record(), nw(m->layers[0].qkv, kAll));
    if (e != cudaSuccess) return cuda_error(e, "embed launch");

    // batch 1-2: the GEMVs stream the tile stream copy of the weights (stream_gemv_launch);
    // batch 3-32: the same copy, batched (batched_gemv_launch); above: row-major passes
    const bool streamed = !m->hmats.empty() && (B <= kPersistMaxBatch || (m->batched_ok && B <= 32));
    int gemv_k = 0;   // GEMV launches so far (their trace rows)
    auto sg = [&](const PMat& M, int epi, bool rms, const float* xf, const __half* x16, const float* nw, void* y,
                  int ld, NextWeights next, int grid = 0, const float* ssq_in = nullptr,
                  const float* w_next = nullptr) {
        StreamGemvArgs ga = {};
        ga.next = next;
        ga.grid = grid;
        // batch 3-32: the RMSNorm folded into the merges (a residual GEMV given the next norm's
        // weight produces its input; an RMSNorm'd GEMV given the sums consumes it)
        ga.ssq_in = ssq_in;
        ga.w_next = w_next;
        ga.ssq_out = w_next ? m->ssq : nullptr;
        if (m->trace) ga.trace = m->trace + (size_t)gemv_k * num_sms() * persist_trace_words();
        unsigned long long* mt =
            m->mtrace ? m->mtrace + (size_t)gemv_k * num_sms() * kMergeTraceWords : nullptr;
        ++gemv_k;
        ga.M = M;
        ga.batch = B;
        ga.epilogue = epi;
        ga.rms = rms ? 1 : 0;
        ga.xf = xf;
        ga.x16 = x16;
        ga.norm_w = nw;
        ga.eps = d.eps;
        ga.y = y;
        ga.ld = ld;
        ga.keys = m->keys;
        ga.active = a->active;
        ga.sync = m->ssync;
        ga.xn = m->xn;
        ga.workspace = m->bws;
        ga.workspace_bytes = m->bws_bytes;
        return B <= kPersistMaxBatch ? stream_gemv_launch(ga, s, pdl) : batched_gemv_launch_traced(ga, mt, s, pdl);
    };
    for (int li = 0; li < d.n_layers; ++li) {
        const ql_layer_desc& L = m->layers[li];
        if (streamed) {
            const PMat* Ms = &m->hmats[4 * li];
            const int qkv_ld = (int)((d.n_heads + 2 * d.n_kv_heads) * d.head_dim);
            // each GEMV warms L2 with the norm weights that the kernel after it reads first
            const NextWeights qk_norms = {{L.q_norm, L.k_norm}, {(size_t)hd * 4, (size_t)hd * 4}};
            const NextWeights ffn_norm = {{L.ffn_norm, nullptr}, {(size_t)d.hidden * 4, 0}};
            const float* next_norm = li + 1 < d.n_layers ? m->layers[li + 1].attn_norm : d.final_norm;
            const NextWeights next_attn_norm = {{next_norm, nullptr}, {(size_t)d.hidden * 4, 0}};
            const NextWeights none = {{nullptr, nullptr}, {0, 0}};
            // batch 3-32: from layer 1 on, the previous down GEMV's merge has written this GEMV's
            // input (f16 x w) and the sums of squares of x (the RMSNorm folded into the merges)
            const bool fold = B > kPersistMaxBatch;
            if ((rc = sg(Ms[0], QL_EPI_NONE, true, m->x, nullptr, L.attn_norm, m->qkv, qkv_ld, qk_norms, 0,
                         fold && li > 0 ? m->ssq : nullptr)) != QL_OK)
                return rc;
            AttnArgs at = {};
            at.qkv = m->qkv;
            at.q_norm = L.q_norm;
            at.k_norm = L.k_norm;
            at.cos_t = m->cos_t;
            at.sin_t = m->sin_t;
            at.eps = d.eps;
            at.max_position = d.max_blocks_per_seq * d.block_size;
            if (kvq) at.kvq = static_cast<uint8_t*>(d.kvq_pool) + kvq_layer * li;
            else {
                at.k_pool = static_cast<__half*>(d.k_pool) + layer_pool * li;
                at.v_pool = static_cast<__half*>(d.v_pool) + layer_pool * li;
            }
            at.block_tables = a->block_tables;
            at.positions = a->positions;
            at.active = a->active;
            at.batch = B;
            at.n_heads = nh;
            at.n_kv_heads = nkv;
            at.head_dim = hd;
            at.block_size = d.block_size;
            at.max_blocks_per_seq = d.max_blocks_per_seq;
            at.num_blocks = d.num_blocks;
            at.scale = 1.0f / sqrtf((float)hd);
            at.out = m->attn;
            at.workspace = m->attn_ws;
            at.workspace_bytes = m->attn_ws_bytes;
            if (m->trace) {   // attention rows follow the GEMV rows
                at.trace = m->trace + (size_t)(4 * d.n_layers + 1 + li) * num_sms() * persist_trace_words();
                at.trace_ctas = num_sms();
            }
            if ((rc = attn_launch(at, s, pdl)) != QL_OK) return rc;
            // the o GEMV leaves out one SM per attention merge (one CTA per sequence and kv head
            // merges the splits, ending after the others): every o CTA then starts on an SM
            // freed early, while the CTA with the most tiles keeps the same count
            const int o_grid = o_gemv_grid(num_sms(), B * nkv, (int)Ms[1].ntile);
            if ((rc = sg(Ms[1], QL_EPI_ADD_RESIDUAL, false, nullptr, m->attn, nullptr, m->x, (int)d.hidden,
                         ffn_norm, o_grid, nullptr, fold && d.num_experts == 0 ? L.ffn_norm : nullptr)) != QL_OK)
                return rc;
            if (d.num_experts > 0) {
                // routed experts: router + top-k, gate|up of the selected experts (RMSNorm'd x,
                // SiLU*up), their down rows against each one's own activations, the combine
                const int64_t K = d.topk, mi = d.moe_inter;
                MoeRouterArgs ra = {};
                ra.x = m->x;
                ra.norm_w = L.ffn_norm;
                ra.router = L.router;
                ra.hidden = (int)d.hidden;
                ra.num_experts = (int)d.num_experts;
                ra.topk = (int)K;
                ra.norm_topk = d.norm_topk;
                ra.eps = d.eps;
                ra.logits = m->mlog;
                ra.ticket = m->mticket;
                ra.eidx = m->meidx;
                ra.ewt = m->mewt;
                if ((rc = moe_router_launch(ra, s, pdl)) != QL_OK) return rc;
                if ((rc = sg(Ms[2], QL_EPI_SILU_MUL, true, m->x, nullptr, L.ffn_norm, m->mact, (int)(K * mi),
                             none)) != QL_OK)
                    return rc;
                if ((rc = sg(Ms[3], QL_EPI_NONE, false, nullptr, m->mact, nullptr, m->medn, (int)(K * d.hidden),
                             none)) != QL_OK)
                    return rc;
                if ((rc = moe_combine_launch(m->x, m->medn, m->mewt, (int)d.hidden, (int)K, s, pdl)) != QL_OK)
                    return rc;
                continue;
            }
            if ((rc = sg(Ms[2], QL_EPI_SILU_MUL, true, m->x, nullptr, L.ffn_norm, m->act, (int)d.intermediate,
                         none, 0, fold ? m->ssq : nullptr)) != QL_OK)
                return rc;
            if ((rc = sg(Ms[3], QL_EPI_ADD_RESIDUAL, false, nullptr, m->act, nullptr, m->x, (int)d.hidden,
                         next_attn_norm, 0, nullptr, fold ? next_norm : nullptr)) != QL_OK)
                return rc;
            continue;
        }
        GemvArgs g = {};
        g.batch = B;
        // qkv projection with the attention RMSNorm as prologue
        g.scales = static_cast<const __half*>(L.qkv.scales);
        g.quants = static_cast<const uint8_t*>(L.qkv.quants);
        g.rows = L.qkv.rows;
        g.cols = L.qkv.cols;
        g.prologue = kProRmsF32;
        g.xf = m->x;
        g.norm_w = L.attn_norm;
        g.eps = d.eps;
        g.epilogue = QL_EPI_NONE;
        g.y_dtype = QL_DTYPE_F32;
        g.y = m->qkv;
        g.next = nw(L.gate_up, kAll);
        if ((rc = gemv_launch(g, s, pdl)) != QL_OK) return rc;

        // attention with the qk-norm + RoPE + KV append fused in (reads the f32 qkv projection)
        AttnArgs at = {};
        at.q = nullptr;
        at.qkv = m->qkv;
        at.q_norm = L.q_norm;
        at.k_norm = L.k_norm;
        at.cos_t = m->cos_t;
        at.sin_t = m->sin_t;
        at.eps = d.eps;
        at.max_position = d.max_blocks_per_seq * d.block_size;
        if (kvq) at.kvq = static_cast<uint8_t*>(d.kvq_pool) + kvq_layer * li;
        else {
            at.k_pool = static_cast<__half*>(d.k_pool) + layer_pool * li;
            at.v_pool = static_cast<__half*>(d.v_pool) + layer_pool * li;
        }
        at.block_tables = a->block_tables;
        at.context_lens = nullptr;
        at.positions = a->positions;
        at.active = a->active;
        at.batch = B;
        at.n_heads = nh;
        at.n_kv_heads = nkv;
        at.head_dim = hd;
        at.block_size = d.block_size;
        at.max_blocks_per_seq = d.max_blocks_per_seq;
        at.num_blocks = d.num_blocks;
        at.scale = 1.0f / sqrtf((float)hd);
        at.out = m->attn;
        at.workspace = m->attn_ws;
        at.workspace_bytes = m->attn_ws_bytes;
        if ((rc = attn_launch(at, s, pdl)) != QL_OK) return rc;

        GemvArgs go = {};
        go.batch = B;
        go.scales = static_cast<const __half*>(L.o.scales);
        go.quants = static_cast<const uint8_t*>(L.o.quants);
        go.rows = L.o.rows;
        go.cols = L.o.cols;
        go.prologue = kProX16;
        go.x16 = m->attn;
        go.epilogue = QL_EPI_ADD_RESIDUAL;
        go.y_dtype = QL_DTYPE_F32;
        go.y = m->x;
        go.residual = m->x;
        if ((rc = gemv_launch(go, s, pdl)) != QL_OK) return rc;

        GemvArgs gu = {};
        gu.batch = B;
        gu.scales = static_cast<const __half*>(L.gate_up.scales);
        gu.quants = static_cast<const uint8_t*>(L.gate_up.quants);
        gu.rows = L.gate_up.rows;
        gu.cols = L.gate_up.cols;
        gu.prologue = kProRmsF32;
        gu.xf = m->x;
        gu.norm_w = L.ffn_norm;
        gu.eps = d.eps;
        gu.epilogue = QL_EPI_SILU_MUL;
        gu.y_dtype = QL_DTYPE_F16;
        gu.y = m->act;
        gu.next = nw(L.down, kAll);
        if ((rc = gemv_launch(gu, s, pdl)) != QL_OK) return rc;

        GemvArgs gd = {};
        gd.batch = B;
        gd.scales = static_cast<const __half*>(L.down.scales);
        gd.quants = static_cast<const uint8_t*>(L.down.quants);
        gd.rows = L.down.rows;
        gd.cols = L.down.cols;
        gd.prologue = kProX16;
        gd.x16 = m->act;
        gd.epilogue = QL_EPI_ADD_RESIDUAL;
        gd.y_dtype = QL_DTYPE_F32;
        gd.y = m->x;
        gd.residual = m->x;
        gd.next = li + 1 < d.n_layers ? nw(m->layers[li + 1].qkv, kAll) : nw(d.lm_head, kLmHead);
        if ((rc = gemv_launch(gd, s, pdl)) != QL_OK) return rc;
    }

    if (streamed) {
        const NextWeights first_norm = {{m->layers[0].attn_norm, nullptr}, {(size_t)d.hidden * 4, 0}};
        // batch 3-32: the last down GEMV's merge wrote f16(x final_norm) and the sums of squares
        const bool fold_lm = B > kPersistMaxBatch && d.num_experts == 0;
        if ((rc = sg(m->hmats.back(), kEpiArgmax, true, m->x, nullptr, d.final_norm,
                     a->logits ? a->logits : m->logits, (int)d.vocab, first_norm, 0,
                     fold_lm ? m->ssq : nullptr)) != QL_OK)
            return rc;
        e = launch(finalize_kernel, dim3(1), dim3(64), 0, s, pdl, m->keys, a->active, a->positions,
                   a->next_tokens, a->out_tokens, (long long)a->out_stride, (float*)nullptr, B);
        if (e != cudaSuccess) return cuda_error(e, "finalize launch");
        return QL_OK;
    }
    GemvArgs gl = {};
    gl.batch = B;
    gl.scales = static_cast<const __half*>(d.lm_head.scales);
    gl.quants = static_cast<const uint8_t*>(d.lm_head.quants);
    gl.rows = d.lm_head.rows;
    gl.cols = d.lm_head.cols;
    gl.prologue = kProRmsF32;
    gl.xf = m->x;
    gl.norm_w = d.final_norm;
    gl.eps = d.eps;
    gl.epilogue = kEpiArgmax;
    gl.y_dtype = QL_DTYPE_F32;
    gl.y = a->logits ? a->logits : m->logits;
    gl.argmax_keys = m->keys;
    gl.active = a->active;
    if ((rc = gemv_launch(gl, s, pdl)) != QL_OK) return rc;

    e = launch(finalize_kernel, dim3(1), dim3(64), 0, s, pdl, m->keys, a->active, a->positions,
               a->next_tokens, a->out_tokens, (long long)a->out_stride, (float*)nullptr, B);
    if (e != cudaSuccess) return cuda_error(e, "finalize launch");
    return QL_OK;
}

// A chunk of T prompt tokens of one sequence through every layer together: the step's GEMVs at
// batch T (stream form at T <= 2, the split-K tensor-core form at 3..32) or, above 32 tokens,
// the tcgen05 GEMM (ql_gemm.cu) after an RMSNorm launch, qk-norm + RoPE + append for all T
// positions, then causal attention of each token over the cache (its own context length), and
// logits of the last token only.
int run_prefill(ql_model* m, const int32_t* tokens, int T, int32_t* position, const int32_t* block_table,
                float* logits, int32_t* next_token, cudaStream_t s) {
    const ql_model_desc& d = m->d;
    const bool pdl = true;
    const int hd = (int)d.head_dim, nh = (int)d.n_heads, nkv = (int)d.n_kv_heads;
    const size_t layer_pool = (size_t)d.num_blocks * nkv * d.block_size * hd;
    const int maxb = (int)d.max_blocks_per_seq;
    int rc;
    cudaError_t e = launch(prefill_setup_kernel, dim3(1), dim3(256), 0, s, pdl, position, block_table, maxb, T, m->pbt,
                           m->ppos, m->plen);
    if (e != cudaSuccess) return cuda_error(e, "prefill setup launch");
    const NextWeights none = {{nullptr, nullptr}, {0, 0}};
    e = launch(embed_kernel, dim3(T), dim3(256), 0, s, pdl, d.embed, tokens, (const int32_t*)nullptr, m->x,
               (int)d.hidden, (int)d.vocab, device_error_record(), none);
    if (e != cudaSuccess) return cuda_error(e, "embed launch");
    auto sg = [&](const PMat& M, int epi, bool rms, const float* xf, const __half* x16, const float* nw, void* y,
                  int ld, int batch) {
        StreamGemvArgs ga = {};
        ga.next = none;
        ga.M = M;
        ga.batch = batch;
        ga.epilogue = epi;
        ga.rms = rms ? 1 : 0;
        ga.xf = xf;
        ga.x16 = x16;
        ga.norm_w = nw;
        ga.eps = d.eps;
        ga.y = y;
        ga.ld = ld;
        ga.keys = m->keys;
        ga.active = nullptr;
        ga.sync = m->ssync;
        ga.xn = m->xn;
        ga.workspace = m->bws;
        ga.workspace_bytes = m->bws_bytes;
        if (batch > kPrefillGemvMax) {   // a GEMM: the normalised input once, then the tcgen05 kernel
            const __half* xin = x16;
            if (rms) {
                if (int rc0 = rms_norm_launch(xf, M.nblk * 32, d.eps, nw, m->xn, batch, s, pdl)) return rc0;
                xin = m->xn;
            }
            GemmArgs g = {};
            g.M = M;
            g.T = batch;
            g.x16 = xin;
            g.y = y;
            g.ld = ld;
            g.epi = epi;
            g.part = static_cast<float*>(m->gws);
            g.part_bytes = m->gws_bytes;
            return gemm_tc_launch(g, s, pdl);
        }
        return batch <= kPersistMaxBatch ? stream_gemv_launch(ga, s, pdl) : batched_gemv_launch(ga, s, pdl);
    };
    const int qkv_ld = (int)((d.n_heads + 2 * d.n_kv_heads) * d.head_dim);
    for (int li = 0; li < d.n_layers; ++li) {
        const ql_layer_desc& L = m->layers[li];
        const PMat* Ms = &m->hmats[4 * li];
        if ((rc = sg(Ms[0], QL_EPI_NONE, true, m->x, nullptr, L.attn_norm, m->qkv, qkv_ld, T)) != QL_OK) return rc;
        RopeArgs ra = {};
        ra.qkv = m->qkv;
        ra.q_norm = L.q_norm;
        ra.k_norm = L.k_norm;
        ra.cos_t = m->cos_t;
        ra.sin_t = m->sin_t;
        ra.positions = m->ppos;
        ra.eps = d.eps;
        ra.batch = T;
        ra.n_heads = nh;
        ra.n_kv_heads = nkv;
        ra.head_dim = hd;
        ra.q_out = m->q16;
        ra.k_pool = static_cast<__half*>(d.k_pool) + layer_pool * li;
        ra.v_pool = static_cast<__half*>(d.v_pool) + layer_pool * li;
        ra.block_tables = m->pbt;
        ra.max_blocks_per_seq = maxb;
        ra.block_size = d.block_size;
        ra.num_blocks = d.num_blocks;
        ra.max_position = d.max_blocks_per_seq * d.block_size;
        if ((rc = rope_launch(ra, s, pdl)) != QL_OK) return rc;
        // the chunk's T tokens against the cache in one pass (each K/V block read once)
        ChunkAttnArgs ca = {};
        ca.q = m->q16;
        ca.k_pool = ra.k_pool;
        ca.v_pool = ra.v_pool;
        ca.block_table = m->pbt;   // row 0: the sequence's table
        ca.position = m->ppos;     // [0] = the chunk's first position
        ca.T = T;
        ca.n_heads = nh;
        ca.n_kv_heads = nkv;
        ca.head_dim = hd;
        ca.max_blocks_per_seq = maxb;
        ca.num_blocks = (int)d.num_blocks;
        ca.scale = 1.0f / sqrtf((float)hd);
        ca.out = m->attn;
        ca.workspace = m->cws;
        ca.workspace_bytes = m->cws_bytes;
        if ((rc = chunk_attn_launch(ca, s, pdl)) != QL_OK) return rc;
        if ((rc = sg(Ms[1], QL_EPI_ADD_RESIDUAL, false, nullptr, m->attn, nullptr, m->x, (int)d.hidden, T)) != QL_OK)
            return rc;
        if ((rc = sg(Ms[2], QL_EPI_SILU_MUL, true, m->x, nullptr, L.ffn_norm, m->act, (int)d.intermediate, T)) != QL_OK)
            return rc;
        if ((rc = sg(Ms[3], QL_EPI_ADD_RESIDUAL, false, nullptr, m->act, nullptr, m->x, (int)d.hidden, T)) != QL_OK)
            return rc;
    }
    // the last token's logits and greedy next token
    if ((rc = sg(m->hmats.back(), kEpiArgmax, true, m->x + (size_t)(T - 1) * d.hidden, nullptr, d.final_norm,
                 logits ? logits : m->logits, (int)d.vocab, 1)) != QL_OK)
        return rc;
    e = launch(prefill_finish_kernel, dim3(1), dim3(32), 0, s, pdl, m->keys, position, next_token, T);
    if (e != cudaSuccess) return cuda_error(e, "prefill finish launch");
    return QL_OK;
}

PMat pmat(const ql_q4_0_matrix& w, bool silu) {
    PMat p = {};
    p.stream = nullptr;
    p.quants = static_cast<const uint8_t*>(w.quants);
    p.scales = static_cast<const __half*>(w.scales);
    p.rows = (int)w.rows;
    p.nblk = (int)(w.cols / 32);
    p.silu = silu ? 1 : 0;
    p.ntile = silu ? (int)((w.rows / 2 + 7) / 8) : (int)((w.rows + 15) / 16);
    return p;
}

// Enable the persistent step kernel when the shape and the device allow it (persist_max_b > 0).
// A shape it does not take is not an error: the step then always runs as separate launches.
int setup_persist(ql_model* m) {
    const ql_model_desc& d = m->d;
    auto al = [](const void* q, uintptr_t n) { return (reinterpret_cast<uintptr_t>(q) & (n - 1)) == 0; };
    auto mat_ok = [&](const ql_q4_0_matrix& w) {
        return w.cols % 128 == 0 && w.rows < (1ll << 30) && al(w.quants, 16) && al(w.scales, 8);
    };
    const bool moe = d.num_experts > 0;
    bool ok = d.vocab < (1ll << 30) && al(d.embed, 16) && al(d.final_norm, 16) && mat_ok(d.lm_head);
    for (const ql_layer_desc& L : m->layers)
        ok = ok && mat_ok(L.qkv) && mat_ok(L.o) && al(L.attn_norm, 16) && al(L.ffn_norm, 16) &&
             (moe ? (mat_ok(L.experts_gate_up) && mat_ok(L.experts_down) && al(L.router, 16))
                  : (mat_ok(L.gate_up) && mat_ok(L.down)));
    if (!ok) return QL_OK;
    const int64_t widths[3] = {d.hidden, moe ? d.moe_inter : d.intermediate, d.n_heads * d.head_dim};
    int64_t w = 0;
    for (int64_t v : widths) w = v > w ? v : w;
    m->max_nblk = (int)(w / 32);
    const int G = (int)(d.n_heads / d.n_kv_heads);
    int maxb = (int)(d.max_batch < kPersistMaxBatch ? d.max_batch : kPersistMaxBatch);
    for (; maxb >= 1; --maxb)
        if (persist_prepare(maxb, m->max_nblk, (int)d.head_dim, G, (int)d.n_layers) == QL_OK) break;
    if (maxb < 1) return QL_OK;
    if (int rc0 = stream_gemv_prepare()) return rc0;
    m->batched_ok = !moe && d.max_batch > kPersistMaxBatch && batched_gemv_shape_ok((int)(d.hidden / 32)) &&
                    batched_gemv_shape_ok((int)(d.intermediate / 32)) &&
                    batched_gemv_shape_ok((int)(d.n_heads * d.head_dim / 32)) && batched_gemv_prepare() == QL_OK;

    std::vector<PLayer> hl(m->layers.size());
    std::vector<PMat> all;     // the step's matrices: 4 per layer, then lm_head
    std::vector<PMat> packs;   // what is re-laid, in stream order (routed experts: one per expert)
    std::vector<size_t> where; // index into packs of each entry of all
    auto add = [&](const PMat& pm) {
        where.push_back(packs.size());
        packs.push_back(pm);
        all.push_back(pm);
    };
    const int64_t mi = d.moe_inter, E = d.num_experts, K = d.topk;
    for (size_t i = 0; i < hl.size(); ++i) {
        const ql_layer_desc& L = m->layers[i];
        add(pmat(L.qkv, false));
        add(pmat(L.o, false));
        if (moe) {
            // gate|up: each expert's 2 mi rows re-laid as its own SiLU*up matrix (8 gate rows and
            // the matching 8 up rows per tile), the experts back to back; the step reads a virtual
            // matrix of the topk selected experts (PMat::sel)
            const int nb1 = (int)(d.hidden / 32);
            where.push_back(packs.size());
            for (int64_t e = 0; e < E; ++e) {
                ql_q4_0_matrix sub = L.experts_gate_up;
                sub.rows = 2 * mi;
                sub.quants = static_cast<const uint8_t*>(L.experts_gate_up.quants) + (size_t)e * 2 * mi * nb1 * 16;
                sub.scales = static_cast<const __half*>(L.experts_gate_up.scales) + (size_t)e * 2 * mi * nb1;
                packs.push_back(pmat(sub, true));
            }
            PMat v1 = pmat(L.experts_gate_up, true);
            v1.rows = (int)(K * 2 * mi);
            v1.ntile = (int)(K * (mi / 8));
            v1.sel = m->meidx;
            v1.etiles = (int)(mi / 8);
            v1.nexp = (int)E;
            v1.nsel = (int)K;
            all.push_back(v1);
            // down: the experts' rows in order are already one matrix; the step reads the topk
            // selected experts' tiles, each against its own activation column
            where.push_back(packs.size());
            packs.push_back(pmat(L.experts_down, false));
            PMat v2 = pmat(L.experts_down, false);
            v2.rows = (int)(K * d.hidden);
            v2.ntile = (int)(K * (d.hidden / 16));
            v2.sel = m->meidx;
            v2.etiles = (int)(d.hidden / 16);
            v2.nexp = (int)E;
            v2.nsel = (int)K;
            v2.xsel = 1;
            all.push_back(v2);
        } else {
            add(pmat(L.gate_up, true));
            add(pmat(L.down, false));
        }
        hl[i].attn_norm = L.attn_norm;
        hl[i].ffn_norm = L.ffn_norm;
        hl[i].q_norm = L.q_norm;
        hl[i].k_norm = L.k_norm;
    }
    add(pmat(d.lm_head, false));
    size_t stream_bytes = 0;
    for (const PMat& pm : packs) stream_bytes += persist_stream_bytes(pm);
    int nsplit = num_sms();
    nsplit = nsplit > 256 ? 256 : nsplit;
    nsplit = nsplit > d.max_blocks_per_seq ? (int)d.max_blocks_per_seq : nsplit;
    m->persist_nsplit = nsplit < 1 ? 1 : nsplit;
    const size_t parts = (size_t)maxb * d.n_heads * m->persist_nsplit;
    int rc = QL_OK;
    auto A = [&](void** p, size_t bytes) { if (rc == QL_OK) rc = alloc(m, p, bytes); };
    A((void**)&m->pstreams, stream_bytes);
    A((void**)&m->players, hl.size() * sizeof(PLayer));
    A((void**)&m->ppm, parts * 4);
    A((void**)&m->ppl, parts * 4);
    A((void**)&m->ppacc, parts * d.head_dim * 4);
    A((void**)&m->ptickets, (size_t)maxb * d.n_kv_heads * 4);
    A((void**)&m->psync, 16);
    A((void**)&m->ssync, 16);
    A((void**)&m->xn, (size_t)d.max_batch * d.hidden * 2);
    A((void**)&m->ssq, (size_t)(d.hidden / 32 + 1) * 32 * sizeof(float));
    if (rc != QL_OK) return rc;
    // the weights re-laid into the tile stream layout that the persistent kernel copies from
    if ((rc = persist_pack_streams(packs.data(), (int)packs.size(), m->pstreams, nullptr)) != QL_OK) return rc;
    for (size_t i = 0; i < all.size(); ++i) all[i].stream = packs[where[i]].stream;
    for (size_t i = 0; i < hl.size(); ++i)
        for (int k = 0; k < 4; ++k) hl[i].m[k] = all[4 * i + k];
    m->plm = all.back();
    m->hmats = all;
    if (d.max_batch > kPrefillGemvMax) {   // the prompt GEMM's K parts (up to 4, the lm_head excluded)
        const int64_t tmax = d.max_batch < kPrefillMax ? d.max_batch : kPrefillMax;
        size_t rmax = 0;
        for (size_t i = 0; i + 1 < all.size(); ++i)
            if (!all[i].silu && (size_t)all[i].ntile * 16 > rmax) rmax = (size_t)all[i].ntile * 16;
        m->gws_bytes = 4 * (size_t)tmax * rmax * sizeof(float);
        A(&m->gws, m->gws_bytes);
        if (rc != QL_OK) return rc;
    }
    if (m->batched_ok) {
        for (const PMat& pm : all) {
            const size_t need = batched_gemv_workspace_bytes(pm.rows, pm.nblk, pm.silu);
            m->bws_bytes = need > m->bws_bytes ? need : m->bws_bytes;
        }
        A(&m->bws, m->bws_bytes);
        if (rc != QL_OK) return rc;
        // the tcgen05 form's row-block tickets start at zero (each call leaves them zero)
        if (cudaMemset(m->bws, 0, m->bws_bytes) != cudaSuccess) return set_error(QL_ECUDA, "ql_model_create: memset");
    }
    cudaError_t e = cudaMemcpy(m->players, hl.data(), hl.size() * sizeof(PLayer), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemset(m->ptickets, 0, (size_t)maxb * d.n_kv_heads * 4);
    if (e == cudaSuccess) e = cudaMemset(m->psync, 0, 16);
    if (e == cudaSuccess) e = cudaMemset(m->ssync, 0, 16);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_error(e, "ql_model_create: persistent step workspace");
    m->persist_stream_bytes = stream_bytes;
    m->persist_max_b = maxb;
    return QL_OK;
}

int check_step_args(ql_model* m, const ql_step_args* a) {
    if (!m || !a) return set_error(QL_EINVAL, "decode step: null model or args");
    if (a->batch < 1 || a->batch > m->d.max_batch)
        return set_error(QL_EINVAL, "decode step: batch must be in [1, max_batch]");
    if (!a->tokens || !a->positions || !a->block_tables || !a->next_tokens)
        return set_error(QL_EINVAL, "decode step: tokens, positions, block_tables and next_tokens are required");
    if (a->out_tokens && a->out_stride <= 0)
        return set_error(QL_EINVAL, "decode step: out_stride must be positive with out_tokens");
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev != m->device) return set_error(QL_EINVAL, "decode step: current device differs from the model's");
    return QL_OK;
}

}  // namespace
}  // namespace ql

using namespace ql;

extern "C" int ql_model_create(const ql_model_desc* desc, ql_model** out) {
    if (!desc || !out) return set_error(QL_EINVAL, "ql_model_create: null pointer");
    *out = nullptr;
    const ql_model_desc& d = *desc;
    QL_REQUIRE(d.hidden > 0 && d.hidden % 32 == 0, "ql_model_create: hidden must be a positive multiple of 32");
    QL_REQUIRE(d.n_layers > 0 && d.layers, "ql_model_create: need layers");
    QL_REQUIRE(d.head_dim == 64 || d.head_dim == 128, "ql_model_create: head_dim must be 64 or 128");
    QL_REQUIRE(d.n_kv_heads > 0 && d.n_heads % d.n_kv_heads == 0, "ql_model_create: bad head counts");
    const int64_t G = d.n_heads / d.n_kv_heads;
    QL_REQUIRE(G == 1 || G == 2 || G == 4 || G == 8, "ql_model_create: GQA group must be 1, 2, 4 or 8");
    QL_REQUIRE(d.num_experts > 0 || (d.intermediate > 0 && d.intermediate % 32 == 0),
               "ql_model_create: intermediate must be a multiple of 32");
    QL_REQUIRE((d.n_heads * d.head_dim) % 32 == 0, "ql_model_create: n_heads*head_dim must be a multiple of 32");
    QL_REQUIRE(d.vocab > 0 && d.embed && d.final_norm, "ql_model_create: need vocab, embed, final_norm");
    QL_REQUIRE(d.block_size == 16, "ql_model_create: block_size must be 16");
    QL_REQUIRE(d.kv_format == QL_KV_F16 || d.kv_format == QL_KV_Q8_0_Q5_1, "ql_model_create: unknown kv_format");
    QL_REQUIRE(d.num_blocks > 0 && (d.kv_format == QL_KV_F16 ? (d.k_pool && d.v_pool) : d.kvq_pool != nullptr),
               "ql_model_create: need KV pools (k_pool and v_pool, or kvq_pool for the quantised format)");
    QL_REQUIRE(d.kv_format == QL_KV_F16 || (reinterpret_cast<uintptr_t>(d.kvq_pool) & 15) == 0,
               "ql_model_create: kvq_pool must be 16-byte aligned");
    QL_REQUIRE(d.max_batch >= 1 && d.max_batch <= 4096, "ql_model_create: max_batch out of range");
    QL_REQUIRE(d.max_blocks_per_seq >= 1, "ql_model_create: bad max_blocks_per_seq");
    QL_REQUIRE(d.eps > 0.f && d.rope_theta > 0.0, "ql_model_create: eps and rope_theta must be positive");
    QL_REQUIRE(check_matrix(d.lm_head, d.vocab, d.hidden), "ql_model_create: lm_head must be [vocab, hidden]");
    const int64_t qkv_rows = (d.n_heads + 2 * d.n_kv_heads) * d.head_dim;
    const bool moe = d.num_experts > 0;
    if (moe) {
        QL_REQUIRE(d.num_experts <= 512 && d.topk >= 1 && d.topk <= d.num_experts && d.topk <= 64,
                   "ql_model_create: routed experts need 1 <= topk <= num_experts <= 512, topk <= 64");
        QL_REQUIRE(d.moe_inter > 0 && d.moe_inter % 128 == 0 && d.hidden % 128 == 0,
                   "ql_model_create: routed experts need moe_inter and hidden multiples of 128");
    }
    for (int64_t i = 0; i < d.n_layers; ++i) {
        const ql_layer_desc& L = d.layers[i];
        const std::string li = " (layer " + std::to_string(i) + ")";
        QL_REQUIRE(L.attn_norm && L.ffn_norm && L.q_norm && L.k_norm, "ql_model_create: missing norm weights" + li);
        QL_REQUIRE(check_matrix(L.qkv, qkv_rows, d.hidden), "ql_model_create: qkv must be [(nh+2nkv)*hd, hidden]" + li);
        QL_REQUIRE(check_matrix(L.o, d.hidden, d.n_heads * d.head_dim), "ql_model_create: o must be [hidden, nh*hd]" + li);
        if (moe) {
            QL_REQUIRE(L.router, "ql_model_create: routed experts need the router weights" + li);
            QL_REQUIRE(check_matrix(L.experts_gate_up, d.num_experts * 2 * d.moe_inter, d.hidden),
                       "ql_model_create: experts_gate_up must be [num_experts*2*moe_inter, hidden]" + li);
            QL_REQUIRE(check_matrix(L.experts_down, d.num_experts * d.hidden, d.moe_inter),
                       "ql_model_create: experts_down must be [num_experts*hidden, moe_inter]" + li);
            continue;
        }
        QL_REQUIRE(check_matrix(L.gate_up, 2 * d.intermediate, d.hidden), "ql_model_create: gate_up must be [2*inter, hidden]" + li);
        QL_REQUIRE(check_matrix(L.down, d.hidden, d.intermediate), "ql_model_create: down must be [hidden, inter]" + li);
    }
    if (!device_error_record()) return set_error(QL_ECUDA, "ql_model_create: cannot allocate the device error record");
    if (int rc0 = gemv_prepare()) return rc0;
    if (int rc0 = attn_prepare()) return rc0;

    ql_model* m = new (std::nothrow) ql_model();
    if (!m) return set_error(QL_ENOMEM, "ql_model_create: out of host memory");
    m->d = d;
    m->layers.assign(d.layers, d.layers + d.n_layers);
    m->d.layers = m->layers.data();
    cudaGetDevice(&m->device);
    if (const char* ev = std::getenv("QL_NEXT_PREFETCH")) m->next_prefetch = std::atoi(ev) != 0;
    const int64_t B = d.max_batch;
    const int64_t max_pos = d.max_blocks_per_seq * d.block_size;
    int rc = QL_OK;
    auto A = [&](void** p, size_t bytes) { if (rc == QL_OK) rc = alloc(m, p, bytes); };
    A((void**)&m->x, B * d.hidden * 4);
    A((void**)&m->qkv, B * qkv_rows * 4);
    A((void**)&m->q16, B * d.n_heads * d.head_dim * 2);
    A((void**)&m->attn, B * d.n_heads * d.head_dim * 2);
    A((void**)&m->act, B * (d.intermediate > 0 ? d.intermediate : 1) * 2);
    A((void**)&m->pbt, B * d.max_blocks_per_seq * 4);
    A((void**)&m->ppos, B * 4);
    A((void**)&m->plen, B * 4);
    if (d.num_experts > 0) {
        A((void**)&m->mlog, d.num_experts * 4);
        A((void**)&m->mticket, 16);
        A((void**)&m->meidx, d.topk * 4);
        A((void**)&m->mewt, d.topk * 4);
        A((void**)&m->mact, d.topk * d.moe_inter * 2);
        A((void**)&m->medn, d.topk * d.hidden * 4);
        if (rc == QL_OK && cudaMemset(m->mticket, 0, 16) != cudaSuccess) rc = set_error(QL_ECUDA, "ql_model_create: memset");
        if (rc == QL_OK && cudaMemset(m->meidx, 0, d.topk * 4) != cudaSuccess) rc = set_error(QL_ECUDA, "ql_model_create: memset");
    }
    A((void**)&m->logits, B * d.vocab * 4);
    A((void**)&m->keys, B * 8);
    A((void**)&m->cos_t, max_pos * (d.head_dim / 2) * 4);
    A((void**)&m->sin_t, max_pos * (d.head_dim / 2) * 4);
    // the split layout depends on the step's batch: size for the largest over 1..max_batch
    for (int64_t b = 1; b <= B; ++b) {
        const size_t need = attn_workspace_bytes(b, (int)d.n_heads, (int)d.n_kv_heads, (int)d.head_dim,
                                                 d.block_size, d.max_blocks_per_seq);
        if (need > m->attn_ws_bytes) m->attn_ws_bytes = need;
    }
    A(&m->attn_ws, m->attn_ws_bytes);
    {   // prefill chunks of up to min(256, max_batch) tokens
        const int tmax = (int)(B < kPrefillMax ? B : kPrefillMax);
        for (int t = 1; t <= tmax; ++t) {
            const size_t need = chunk_attn_workspace_bytes(t, (int)d.n_heads, (int)d.n_kv_heads, (int)d.head_dim);
            if (need > m->cws_bytes) m->cws_bytes = need;
        }
        A(&m->cws, m->cws_bytes);
    }
    if (rc == QL_OK) {
        std::vector<float> hc(max_pos * (d.head_dim / 2)), hs(hc.size());
        rc = ql_rope_tables(hc.data(), hs.data(), max_pos, (int)d.head_dim, d.rope_theta);
        cudaError_t e = cudaSuccess;
        if (rc == QL_OK) e = cudaMemcpy(m->cos_t, hc.data(), hc.size() * 4, cudaMemcpyHostToDevice);
        if (rc == QL_OK && e == cudaSuccess) e = cudaMemcpy(m->sin_t, hs.data(), hs.size() * 4, cudaMemcpyHostToDevice);
        if (rc == QL_OK && e == cudaSuccess) e = cudaMemset(m->keys, 0, B * 8);
        if (rc == QL_OK && e == cudaSuccess) e = cudaMemset(m->attn_ws, 0, m->attn_ws_bytes);
        if (rc == QL_OK && e == cudaSuccess) e = cudaMemset(m->x, 0, B * d.hidden * 4);
        if (rc == QL_OK && e == cudaSuccess) e = cudaDeviceSynchronize();
        if (rc == QL_OK && e != cudaSuccess) rc = cuda_error(e, "ql_model_create: workspace init");
    }
    if (rc == QL_OK) rc = setup_persist(m);
    if (rc != QL_OK) {
        std::string msg = ql_last_error();
        ql_model_destroy(m);
        return set_error(rc, msg);
    }
    *out = m;
    return QL_OK;
}

extern "C" int ql_model_destroy(ql_model* m) {
    if (!m) return QL_OK;
    for (auto& kv : m->graphs) cudaGraphExecDestroy(kv.second);
    for (void* p : m->owned) cudaFree(p);
    delete m;
    return QL_OK;
}

extern "C" int ql_model_set_option(ql_model* m, int option, int64_t value) {
    if (!m) return set_error(QL_EINVAL, "ql_model_set_option: null model");
    switch (option) {
        case QL_OPT_STEP_KERNEL:
            if (value != QL_STEP_AUTO && value != QL_STEP_LAUNCHES && value != QL_STEP_PERSISTENT)
                return set_error(QL_EINVAL, "ql_model_set_option: unknown step kernel");
            if (value == QL_STEP_PERSISTENT && (m->persist_max_b < 1 || m->d.kv_format != QL_KV_F16 || m->d.num_experts > 0))
                return set_error(QL_EINVAL, "ql_model_set_option: the persistent step kernel is not available for this model");
            m->step_kernel = (int)value;
            return QL_OK;
        case QL_OPT_BARRIER_TIMEOUT_NS:
            if (value < 0) return set_error(QL_EINVAL, "ql_model_set_option: negative timeout");
            m->barrier_timeout_ns = (unsigned long long)value;
            return QL_OK;
        case QL_OPT_TEST_BARRIER_EXTRA:
            if (value < 0 || value > 1) return set_error(QL_EINVAL, "ql_model_set_option: extra arrivals must be 0 or 1");
            m->barrier_extra = (unsigned int)value;
            return QL_OK;
        case QL_OPT_STEP_TRACE:
            if ((value & 7) != 0) return set_error(QL_EINVAL, "ql_model_set_option: trace buffer must be 8-byte aligned");
            m->trace = reinterpret_cast<unsigned long long*>(static_cast<uintptr_t>(value));
            return QL_OK;
        case QL_OPT_MERGE_TRACE:
            if ((value & 7) != 0) return set_error(QL_EINVAL, "ql_model_set_option: trace buffer must be 8-byte aligned");
            m->mtrace = reinterpret_cast<unsigned long long*>(static_cast<uintptr_t>(value));
            return QL_OK;
        default:
            return set_error(QL_EINVAL, "ql_model_set_option: unknown option");
    }
}

extern "C" int64_t ql_model_persistent_max_batch(const ql_model* m) { return m ? m->persist_max_b : 0; }

extern "C" int ql_decode_step(ql_model* m, const ql_step_args* args, void* stream) {
    int rc = check_step_args(m, args);
    if (rc != QL_OK) return rc;
    return run_step(m, args, static_cast<cudaStream_t>(stream));
}

extern "C" int ql_prefill_chunk(ql_model* m, const int32_t* d_tokens, int64_t n_tokens, int32_t* d_position,
                                const int32_t* d_block_table, float* d_logits, int32_t* d_next_token, void* stream) {
    if (!m || !d_tokens || !d_position || !d_block_table) return set_error(QL_EINVAL, "ql_prefill_chunk: null pointer");
    const ql_model_desc& d = m->d;
    if (d.num_experts > 0 || d.kv_format != QL_KV_F16)
        return set_error(QL_EINVAL, "ql_prefill_chunk: dense models with the f16 KV cache only");
    if (n_tokens < 1 || n_tokens > kPrefillMax || n_tokens > d.max_batch)
        return set_error(QL_EINVAL, "ql_prefill_chunk: n_tokens must be in [1, min(256, max_batch)]");
    if (m->hmats.empty() || (n_tokens > kPersistMaxBatch && n_tokens <= kPrefillGemvMax && !m->batched_ok))
        return set_error(QL_EINVAL, "ql_prefill_chunk: needs the tile stream copies (and the batched GEMV above 2 tokens)");
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev != m->device) return set_error(QL_EINVAL, "ql_prefill_chunk: current device differs from the model's");
    return run_prefill(m, d_tokens, (int)n_tokens, d_position, d_block_table, d_logits, d_next_token,
                       static_cast<cudaStream_t>(stream));
}

extern "C" int ql_decode_graph_capture(ql_model* m, const ql_step_args* args, void* stream) {
    int rc = check_step_args(m, args);
    if (rc != QL_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!s) return set_error(QL_EINVAL, "ql_decode_graph_capture: needs a non-default stream");
    QL_TRY_CUDA(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal));
    rc = run_step(m, args, s);
    cudaGraph_t g = nullptr;
    cudaError_t e = cudaStreamEndCapture(s, &g);
    if (rc != QL_OK) {
        if (g) cudaGraphDestroy(g);
        return rc;
    }
    if (e != cudaSuccess) return cuda_error(e, "cudaStreamEndCapture");
    cudaGraphExec_t ex = nullptr;
    e = cudaGraphInstantiate(&ex, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) return cuda_error(e, "cudaGraphInstantiate");
    auto it = m->graphs.find(args->batch);
    if (it != m->graphs.end()) cudaGraphExecDestroy(it->second);
    m->graphs[args->batch] = ex;
    m->graph_args[args->batch] = *args;
    return QL_OK;
}

extern "C" int ql_decode_graph_step_host(ql_model* m, int64_t batch, const int32_t* h_tokens, int32_t* h_next_tokens,
                                         void* stream) {
    if (!m) return set_error(QL_EINVAL, "ql_decode_graph_step_host: null model");
    if (!h_tokens || !h_next_tokens) return set_error(QL_EINVAL, "ql_decode_graph_step_host: null host buffer");
    auto it = m->graphs.find(batch);
    if (it == m->graphs.end())
        return set_error(QL_ESTATE, "ql_decode_graph_step_host: no graph captured for batch " + std::to_string(batch));
    const ql_step_args& a = m->graph_args[batch];
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t bytes = (size_t)batch * sizeof(int32_t);
    QL_TRY_CUDA(cudaMemcpyAsync(const_cast<int32_t*>(a.tokens), h_tokens, bytes, cudaMemcpyHostToDevice, s));
    QL_TRY_CUDA(cudaGraphLaunch(it->second, s));
    QL_TRY_CUDA(cudaMemcpyAsync(h_next_tokens, a.next_tokens, bytes, cudaMemcpyDeviceToHost, s));
    QL_TRY_CUDA(cudaStreamSynchronize(s));
    return QL_OK;
}

extern "C" int ql_decode_graph_replay(ql_model* m, int64_t batch, int n_steps, void* stream) {
    if (!m) return set_error(QL_EINVAL, "ql_decode_graph_replay: null model");
    if (n_steps < 0) return set_error(QL_EINVAL, "ql_decode_graph_replay: n_steps < 0");
    auto it = m->graphs.find(batch);
    if (it == m->graphs.end())
        return set_error(QL_ESTATE, "ql_decode_graph_replay: no graph captured for batch " + std::to_string(batch));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (int i = 0; i < n_steps; ++i) QL_TRY_CUDA(cudaGraphLaunch(it->second, s));
    return QL_OK;
}
