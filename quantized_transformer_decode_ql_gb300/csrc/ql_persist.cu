// Persistent decode step: kernels for head_dim 128 and the host entry points (the kernel
// itself is in ql_persist.cuh; head_dim 64 in ql_persist_hd64.cu).
#include "ql_persist.cuh"

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

int stream_gemv_prepare() {
    static std::mutex mu;
    static std::set<int> done;
    int dev = 0;
    QL_TRY_CUDA(cudaGetDevice(&dev));
    std::lock_guard<std::mutex> lk(mu);
    if (done.count(dev)) return QL_OK;
    cudaError_t e = persist::stream_gemv_one<1>(false, nullptr, nullptr, 0, 0, nullptr, false);
    if (e == cudaSuccess) e = persist::stream_gemv_one<2>(false, nullptr, nullptr, 0, 0, nullptr, false);
    if (e != cudaSuccess) return cuda_error(e, "stream gemv: kernel attributes");
    done.insert(dev);
    return QL_OK;
}

int stream_gemv_launch(const StreamGemvArgs& a, cudaStream_t s, bool pdl) {
    QL_REQUIRE(a.M.stream && a.M.nblk > 0 && a.M.nblk % persist::kUnitBlocks == 0, "stream gemv: bad matrix");
    QL_REQUIRE(a.batch == 1 || a.batch == 2, "stream gemv: batch must be 1 or 2");
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
    const size_t smem = persist::kRingBytes + persist::gemv_region_bytes(a.batch, a.M.nblk);
    const cudaError_t e = a.batch == 1 ? persist::stream_gemv_one<1>(true, &p, &g, smem, num_sms(), s, pdl)
                                       : persist::stream_gemv_one<2>(true, &p, &g, smem, num_sms(), s, pdl);
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
