// Persistent decode step: kernels for head_dim 128 and the host entry points (the kernel
// itself is in ql_persist.cuh; head_dim 64 in ql_persist_hd64.cu).
#include "ql_persist.cuh"

#include <atomic>
#include <cstdlib>
#include <map>
#include <mutex>
#include <set>
#include <string>

namespace ql {

cudaError_t persist_dispatch_hd128(int G, bool launch, const PersistParams* p, size_t smem, int grid,
                                   cudaStream_t s, int* occ) {
    return persist::dispatch<128>(G, launch, p, smem, grid, s, occ);
}

size_t persist_smem_bytes(int batch, int max_nblk, int head_dim, int group, int n_layers) {
    return persist::kRingBytes + persist::region_bytes(batch, max_nblk, head_dim, group) +
           persist::mat_table_bytes(n_layers);
}

int persist_prepare(int batch, int max_nblk, int head_dim, int group, int n_layers) {
    QL_REQUIRE(batch >= 1 && batch <= kPersistMaxBatch, "persistent step: batch out of range");
    QL_REQUIRE(head_dim == 64 || head_dim == 128, "persistent step: head_dim must be 64 or 128");
    QL_REQUIRE(group == 1 || group == 2 || group == 4 || group == 8, "persistent step: GQA group must be 1, 2, 4 or 8");
    QL_REQUIRE(max_nblk > 0 && max_nblk % persist::kUnitBlocks == 0,
               "persistent step: matrix widths must be multiples of 128");
    int dev = 0, coop = 0, optin = 0;
    QL_TRY_CUDA(cudaGetDevice(&dev));
    QL_TRY_CUDA(cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev));
    QL_TRY_CUDA(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
    QL_REQUIRE(coop != 0, "persistent step: the device has no cooperative launch");
    const size_t smem = persist_smem_bytes(batch, max_nblk, head_dim, group, n_layers);
    if (smem > (size_t)optin)
        return set_error(QL_EINVAL, "persistent step: needs " + std::to_string(smem) +
                                        " bytes of shared memory per CTA, the device allows " + std::to_string(optin));
    int occ = 0;
    const cudaError_t e = head_dim == 128 ? persist_dispatch_hd128(group, false, nullptr, smem, 0, nullptr, &occ)
                                          : persist_dispatch_hd64(group, false, nullptr, smem, 0, nullptr, &occ);
    if (e != cudaSuccess) return cuda_error(e, "persistent step: kernel attributes");
    QL_REQUIRE(occ >= 1, "persistent step: one CTA per SM does not fit (shared memory or registers)");
    return QL_OK;
}

size_t persist_stream_bytes(const PMat& m) {
    return (size_t)m.ntile * (m.nblk / persist::kUnitBlocks) * persist::kUnitBytes;
}

int persist_pack_streams(PMat* mats, int n, uint8_t* buf, cudaStream_t s) {
    size_t off = 0;
    const int grid = 4 * num_sms();
    for (int i = 0; i < n; ++i) {
        mats[i].stream = buf + off;
        persist::stream_pack_kernel<<<grid, 256, 0, s>>>(mats[i], buf + off);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_error(e, "persistent step: stream pack launch");
        off += persist_stream_bytes(mats[i]);
    }
    return QL_OK;
}

static_assert(persist::kEpiF32 == QL_EPI_NONE && persist::kEpiResid == QL_EPI_ADD_RESIDUAL &&
                  persist::kEpiSilu == QL_EPI_SILU_MUL && persist::kEpiLogits == kEpiArgmax,
              "epilogue codes");

static int stream_gemv_warps() {
    static const int w = [] {
        const char* e = std::getenv("QL_STREAM_GEMV_WARPS");
        return e && std::atoi(e) == 8 ? 8 : 16;
    }();
    return w;
}

// Activation form of the batch 1-2 GEMV (process-wide; graphs keep the form they were captured
// with): 16-bit fixed point per 32-element block (default), or the int8 absmax form of the
// pages ([IL] CudaQwen3::absmax) with QL_GEMV_ACT=int8 or ql_set_gemv_activation_form.
static std::atomic<int> g_act_form{-1};
static int act_form() {
    int f = g_act_form.load();
    if (f < 0) {
        const char* e = std::getenv("QL_GEMV_ACT");
        f = (e != nullptr && std::string(e) == "int8") ? QL_GEMV_ACT_INT8 : QL_GEMV_ACT_INT16;
        int expect = -1;
        g_act_form.compare_exchange_strong(expect, f);
        f = g_act_form.load();
    }
    return f;
}

int stream_gemv_prepare() {
    static std::mutex mu;
    static std::set<int> done;
    int dev = 0;
    QL_TRY_CUDA(cudaGetDevice(&dev));
    std::lock_guard<std::mutex> lk(mu);
    if (done.count(dev)) return QL_OK;
    cudaError_t e = persist::stream_gemv_one<1, 8>(false, nullptr, nullptr, 0, 0, nullptr, false);
    if (e == cudaSuccess) e = persist::stream_gemv_one<2, 8>(false, nullptr, nullptr, 0, 0, nullptr, false);
    if (e == cudaSuccess) e = persist::stream_gemv_one<1, 16>(false, nullptr, nullptr, 0, 0, nullptr, false);
    if (e == cudaSuccess) e = persist::stream_gemv_one<2, 16>(false, nullptr, nullptr, 0, 0, nullptr, false);
    if (e == cudaSuccess) e = persist::stream_gemv_one<1, 16, true>(false, nullptr, nullptr, 0, 0, nullptr, false);
    if (e == cudaSuccess) e = persist::stream_gemv_one<2, 16, true>(false, nullptr, nullptr, 0, 0, nullptr, false);
    if (e == cudaSuccess) e = persist::stream_gemv_one<1, 16, false, true>(false, nullptr, nullptr, 0, 0, nullptr, false);
    if (e != cudaSuccess) return cuda_error(e, "stream gemv: kernel attributes");
    done.insert(dev);
    return QL_OK;
}

int persist_trace_words() { return persist::kTraceWords; }

int stream_gemv_launch(const StreamGemvArgs& a, cudaStream_t s, bool pdl) {
    QL_REQUIRE(a.M.stream && a.M.nblk > 0 && a.M.nblk % persist::kUnitBlocks == 0, "stream gemv: bad matrix");
    QL_REQUIRE(a.batch == 1 || a.batch == 2, "stream gemv: batch must be 1 or 2");
    QL_REQUIRE(!a.M.sel || (a.batch == 1 && a.M.etiles > 0 && a.M.nsel > 0 && a.M.nsel <= 64 && a.M.nexp > 0),
               "stream gemv: routed experts need batch 1 and a valid selection");
    QL_REQUIRE(a.rms ? (a.xf && a.norm_w) : a.x16 != nullptr, "stream gemv: null input");
    QL_REQUIRE(a.y && a.sync, "stream gemv: null output");
    QL_REQUIRE(a.epilogue != kEpiArgmax || a.keys, "stream gemv: argmax needs keys");
    QL_REQUIRE((a.epilogue == QL_EPI_SILU_MUL) == (a.M.silu != 0), "stream gemv: SiLU*up needs a matrix packed for it");
    DevError* err = device_error_record();
    if (!err) return set_error(QL_ECUDA, "stream gemv: no device error record");
    if (int rc = stream_gemv_prepare()) return rc;
    PersistParams p = {};
    p.B = a.batch;
    p.max_nblk = a.M.nblk;
    p.eps = a.eps;
    p.barrier_timeout_ns = 2000000000ull;
    p.keys = a.keys;
    p.active = a.active;
    p.sync = a.sync;
    p.err = err;
    persist::StreamGemv g = {};
    g.M = a.M;
    g.epi = a.epilogue;
    g.rms = a.rms;
    g.xf = a.xf;
    g.x16 = a.x16;
    g.norm_w = a.norm_w;
    g.y = a.y;
    g.ld = a.ld;
    g.trace = stream_gemv_warps() == 16 ? a.trace : nullptr;   // the trace rows hold one CTA per SM
    g.next = a.next;
    // one ring slot per warp before the wait, the other after the activations are staged (their
    // loads then queue behind half as much weight data; measured faster than both slots or none
    // in the decode step); QL_STREAM_PREWAIT=0..2 selects another count for A/B measurements
    static const int prewait = [] {
        const char* e = std::getenv("QL_STREAM_PREWAIT");
        const int v = e ? std::atoi(e) : 1;
        return v < 0 ? 0 : (v > persist::kStages ? persist::kStages : v);
    }();
    // routed experts: which tiles to copy is known only once the predecessor (the router) is
    // done, so nothing is issued before the wait
    g.prewait = a.M.sel ? 0 : prewait;
    // one CTA of 16 warps per SM (measured faster in the step than two CTAs of 8 warps, which
    // would let a kernel's set-up overlap the previous kernel's tail); QL_STREAM_GEMV_WARPS=8
    // selects the two-CTA form for A/B measurements
    const int warps = stream_gemv_warps();
    const int staged = a.M.xsel ? a.M.nsel : a.batch;   // activation columns staged
    const size_t smem = (size_t)warps * persist::kStages * persist::kSlotBytes +
                        persist::gemv_region_bytes(staged, a.M.nblk, warps);
    int grid = num_sms() * (warps == 8 ? 2 : 1);
    if (a.grid > 0 && a.grid < grid) grid = a.grid;
    cudaError_t e;
    if (a.M.sel)   // routed experts (batch 1, 16 warps)
        e = persist::stream_gemv_one<1, 16, false, true>(true, &p, &g, smem, num_sms(), s, pdl);
    else if (act_form() == QL_GEMV_ACT_INT8)   // the int8 absmax form (16 warps)
        e = a.batch == 1 ? persist::stream_gemv_one<1, 16, true>(true, &p, &g, smem, num_sms(), s, pdl)
                         : persist::stream_gemv_one<2, 16, true>(true, &p, &g, smem, num_sms(), s, pdl);
    else if (warps == 8)
        e = a.batch == 1 ? persist::stream_gemv_one<1, 8>(true, &p, &g, smem, grid, s, pdl)
                         : persist::stream_gemv_one<2, 8>(true, &p, &g, smem, grid, s, pdl);
    else
        e = a.batch == 1 ? persist::stream_gemv_one<1, 16>(true, &p, &g, smem, grid, s, pdl)
                         : persist::stream_gemv_one<2, 16>(true, &p, &g, smem, grid, s, pdl);
    if (e != cudaSuccess) return cuda_error(e, "stream gemv launch");
    return QL_OK;
}

int persist_launch(const PersistParams& p, int head_dim, int group, cudaStream_t s) {
    const size_t smem = persist_smem_bytes(p.B, p.max_nblk, head_dim, group, p.n_layers);
    const int grid = num_sms();
    const cudaError_t e = head_dim == 128 ? persist_dispatch_hd128(group, true, &p, smem, grid, s, nullptr)
                                          : persist_dispatch_hd64(group, true, &p, smem, grid, s, nullptr);
    if (e != cudaSuccess) return cuda_error(e, "persistent step launch");
    return QL_OK;
}

}  // namespace ql

// ---------------------------------------------------------------------------------------------
// C ABI: the tile stream layout and the batch 1-2 GEMV over it.
namespace {

// abort flag of the stand-alone GEMV's bounded waits (written only when a wait runs out)
__device__ unsigned int g_stream_gemv_sync[4];

bool stream_shape_ok(int64_t rows, int64_t cols, int silu) {
    return rows > 0 && cols > 0 && cols % 128 == 0 && rows < (1ll << 30) && cols < (1ll << 24) &&
           (!silu || rows % 2 == 0);
}

ql::PMat stream_mat(const void* d_stream, int64_t rows, int64_t cols, int silu) {
    ql::PMat m = {};
    m.stream = static_cast<const uint8_t*>(d_stream);
    m.rows = (int)rows;
    m.nblk = (int)(cols / 32);
    m.silu = silu ? 1 : 0;
    m.ntile = silu ? (int)((rows / 2 + 7) / 8) : (int)((rows + 15) / 16);
    return m;
}

bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; }

}  // namespace

extern "C" int ql_set_gemv_activation_form(int form) {
    using namespace ql;
    QL_REQUIRE(form == QL_GEMV_ACT_INT16 || form == QL_GEMV_ACT_INT8, "ql_set_gemv_activation_form: unknown form");
    const int prev = act_form();
    g_act_form.store(form);
    return prev;
}

extern "C" int64_t ql_q4_0_stream_bytes(int64_t rows, int64_t cols, int silu) {
    if (!stream_shape_ok(rows, cols, silu)) return 0;
    return (int64_t)ql::persist_stream_bytes(stream_mat(nullptr, rows, cols, silu));
}

extern "C" int ql_q4_0_stream_pack(const void* d_scales, const void* d_quants, int64_t rows, int64_t cols,
                                   int silu, void* d_stream, void* stream) {
    using namespace ql;
    QL_REQUIRE(d_scales && d_quants && d_stream, "ql_q4_0_stream_pack: null pointer");
    QL_REQUIRE(stream_shape_ok(rows, cols, silu), "ql_q4_0_stream_pack: need cols % 128 == 0 (and even rows with silu)");
    QL_REQUIRE(aligned(d_quants, 16) && aligned(d_stream, 16) && aligned(d_scales, 8),
               "ql_q4_0_stream_pack: codes and stream must be 16-byte aligned, scales 8-byte");
    PMat m = stream_mat(nullptr, rows, cols, silu);
    m.quants = static_cast<const uint8_t*>(d_quants);
    m.scales = static_cast<const __half*>(d_scales);
    return persist_pack_streams(&m, 1, static_cast<uint8_t*>(d_stream), static_cast<cudaStream_t>(stream));
}

extern "C" int64_t ql_gemv_q4_0_stream_workspace_bytes(int64_t rows, int64_t cols, int silu) {
    using namespace ql;
    if (!stream_shape_ok(rows, cols, silu) || !batched_gemv_shape_ok((int)(cols / 32))) return 0;
    return (int64_t)batched_gemv_workspace_bytes((int)rows, (int)(cols / 32), silu ? 1 : 0);
}

extern "C" int ql_gemv_q4_0_stream(const void* d_stream, int64_t rows, int64_t cols, const void* d_x, int64_t batch,
                                   void* d_y, int epilogue, void* d_workspace, int64_t workspace_bytes,
                                   void* stream) {
    using namespace ql;
    QL_REQUIRE(d_stream && d_x && d_y, "ql_gemv_q4_0_stream: null pointer");
    QL_REQUIRE(epilogue == QL_EPI_NONE || epilogue == QL_EPI_ADD_RESIDUAL || epilogue == QL_EPI_SILU_MUL,
               "ql_gemv_q4_0_stream: unknown epilogue");
    const int silu = epilogue == QL_EPI_SILU_MUL;
    QL_REQUIRE(stream_shape_ok(rows, cols, silu), "ql_gemv_q4_0_stream: need cols % 128 == 0 (and even rows with SiLU*up)");
    QL_REQUIRE(batch >= 1 && batch <= 32, "ql_gemv_q4_0_stream: batch must be in [1, 32]");
    QL_REQUIRE(batch <= 2 || batched_gemv_shape_ok((int)(cols / 32)),
               "ql_gemv_q4_0_stream: batches above 2 need cols in 128..896 or a multiple of 1024");
    QL_REQUIRE(aligned(d_stream, 16) && aligned(d_x, 16) && aligned(d_y, 4),
               "ql_gemv_q4_0_stream: stream and x must be 16-byte aligned, y 4-byte");
    QL_REQUIRE(batch <= 2 || (d_workspace && aligned(d_workspace, 256) && workspace_bytes >= 0),
               "ql_gemv_q4_0_stream: batches above 2 need a 256-byte aligned workspace");
    // the flag's address, resolved once per device (the lookup may load the module lazily,
    // which a stream capture does not allow; the first call should come before any capture)
    static std::mutex mu;
    static std::map<int, void*> addr;
    int dev = 0;
    QL_TRY_CUDA(cudaGetDevice(&dev));
    void* sync = nullptr;
    {
        std::lock_guard<std::mutex> lk(mu);
        auto it = addr.find(dev);
        if (it == addr.end()) {
            QL_TRY_CUDA(cudaGetSymbolAddress(&sync, g_stream_gemv_sync));
            addr[dev] = sync;
        } else {
            sync = it->second;
        }
    }
    StreamGemvArgs a = {};
    a.M = stream_mat(d_stream, rows, cols, silu);
    a.batch = (int)batch;
    a.epilogue = epilogue;
    a.rms = 0;
    a.x16 = static_cast<const __half*>(d_x);
    a.y = d_y;
    a.ld = (int)(silu ? rows / 2 : rows);
    a.sync = static_cast<unsigned int*>(sync);
    a.workspace = d_workspace;
    a.workspace_bytes = (size_t)workspace_bytes;
    return batch <= 2 ? stream_gemv_launch(a, static_cast<cudaStream_t>(stream), true)
                      : batched_gemv_launch(a, static_cast<cudaStream_t>(stream), true);
}
