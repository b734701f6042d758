// Host side of libql: status strings, the thread-local error message, the q4_0 codec,
// RoPE tables, the KV block allocator and the per-device error record.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <functional>
#include <map>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

#include "ql_f16.h"
#include "ql_internal.h"
#include "ql_kvq.h"

namespace ql {

static thread_local std::string g_last_error;

int set_error(int status, const std::string& msg) {
    g_last_error = msg;
    return status;
}

int cuda_error(cudaError_t e, const char* what) {
    return set_error(QL_ECUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" +
                                   cudaGetErrorString(e) + ")");
}

static std::mutex g_dev_mu;
static std::map<int, DevError*> g_dev_err;
static std::map<int, int> g_sms;

DevError* device_error_record() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    auto it = g_dev_err.find(dev);
    if (it != g_dev_err.end()) return it->second;
    DevError* p = nullptr;
    if (cudaMalloc(&p, sizeof(DevError)) != cudaSuccess) return nullptr;
    if (cudaMemset(p, 0, sizeof(DevError)) != cudaSuccess) return nullptr;
    if (cudaDeviceSynchronize() != cudaSuccess) return nullptr;
    g_dev_err[dev] = p;
    return p;
}

DevError* device_error_record_existing() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    auto it = g_dev_err.find(dev);
    return it == g_dev_err.end() ? nullptr : it->second;
}

int num_sms() {
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(g_dev_mu);
    auto it = g_sms.find(dev);
    if (it != g_sms.end()) return it->second;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 1;
    g_sms[dev] = n;
    return n;
}

static const char* where_name(int w) {
    switch (w) {
        case kErrEmbedToken: return "embedding lookup: token id outside the vocabulary";
        case kErrRopePosition: return "KV append: position outside the block table / RoPE table";
        case kErrRopeBlock: return "KV append: block id outside the pool";
        case kErrAttnBlock: return "attention: block id outside the pool";
        case kErrAttnLength: return "attention: context length outside the block table";
        case kErrPackNonFinite: return "q4_0 pack: non-finite weight";
        case kErrPackOverflow: return "q4_0 pack: block scale overflows f16";
        case kErrGemvStage: return "gemv: a staged weight copy did not arrive (bounded wait expired)";
        case kErrStepBarrier: return "persistent step: a grid barrier wait ran out (index = barrier, value = CTA)";
        case kErrKvNonFinite: return "KV row quantiser: non-finite value (index = row, value = block)";
        case kErrKvOverflow: return "KV row quantiser: block scale or minimum overflows f16 (index = row, value = block)";
        default: return "unknown";
    }
}

}  // namespace ql

using namespace ql;

extern "C" {

const char* ql_status_str(int s) {
    switch (s) {
        case QL_OK: return "QL_OK";
        case QL_EINVAL: return "QL_EINVAL";
        case QL_ENOMEM: return "QL_ENOMEM";
        case QL_ECUDA: return "QL_ECUDA";
        case QL_EPOOL: return "QL_EPOOL";
        case QL_ERANGE: return "QL_ERANGE";
        case QL_EDEVICE: return "QL_EDEVICE";
        case QL_ESTATE: return "QL_ESTATE";
        default: return "QL_UNKNOWN";
    }
}

const char* ql_last_error(void) { return g_last_error.c_str(); }

int ql_version(void) { return 1; }

// ------------------------------------------------------------------ quantised KV rows
// The q8_0 (keys) / q5_1 (values) row codecs of ql_kvq.h, on host rows.
int64_t ql_kv_q8_0_row_bytes(int64_t dim) { return dim > 0 ? (dim + 31) / 32 * ql::kQ8Bytes : 0; }
int64_t ql_kv_q5_1_row_bytes(int64_t dim) { return dim > 0 ? (dim + 31) / 32 * ql::kQ5Bytes : 0; }

static int kv_quantize(const char* name, const float* x, int64_t rows, int64_t dim, uint8_t* out,
                       int block_bytes, int (*block)(const float*, int, uint8_t*)) {
    if (!x || !out) return set_error(QL_EINVAL, std::string(name) + ": null pointer");
    if (rows <= 0 || dim <= 0) return set_error(QL_EINVAL, std::string(name) + ": need rows > 0 and dim > 0");
    for (int64_t i = 0; i < rows * dim; ++i)
        if (!std::isfinite(x[i]))
            return set_error(QL_EINVAL, std::string(name) + ": non-finite value in row " + std::to_string(i / dim));
    const int64_t nblk = (dim + 31) / 32, rb = nblk * block_bytes;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < nblk; ++j) {
            const int64_t e0 = j * 32;
            const int n = (int)std::min<int64_t>(32, dim - e0);
            if (block(x + r * dim + e0, n, out + r * rb + j * block_bytes))
                return set_error(QL_EINVAL, std::string(name) + ": a block scale or minimum overflows f16 in row " +
                                                std::to_string(r));
        }
    return QL_OK;
}

int ql_kv_quantize_q8_0(const float* x, int64_t rows, int64_t dim, uint8_t* out) {
    return kv_quantize("ql_kv_quantize_q8_0", x, rows, dim, out, ql::kQ8Bytes, ql::kvq_q8_block);
}

int ql_kv_quantize_q5_1(const float* x, int64_t rows, int64_t dim, uint8_t* out) {
    return kv_quantize("ql_kv_quantize_q5_1", x, rows, dim, out, ql::kQ5Bytes, ql::kvq_q5_block);
}

static int kv_dequantize(const char* name, const uint8_t* in, int64_t rows, int64_t dim, float* x,
                         int block_bytes, float (*value)(const uint8_t*, int)) {
    if (!in || !x) return set_error(QL_EINVAL, std::string(name) + ": null pointer");
    if (rows <= 0 || dim <= 0) return set_error(QL_EINVAL, std::string(name) + ": need rows > 0 and dim > 0");
    const int64_t rb = (dim + 31) / 32 * block_bytes;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t e = 0; e < dim; ++e)
            x[r * dim + e] = value(in + r * rb + (e >> 5) * block_bytes, (int)(e & 31));
    return QL_OK;
}

int ql_kv_dequantize_q8_0(const uint8_t* in, int64_t rows, int64_t dim, float* x) {
    return kv_dequantize("ql_kv_dequantize_q8_0", in, rows, dim, x, ql::kQ8Bytes, ql::kvq_q8_value);
}

int ql_kv_dequantize_q5_1(const uint8_t* in, int64_t rows, int64_t dim, float* x) {
    return kv_dequantize("ql_kv_dequantize_q5_1", in, rows, dim, x, ql::kQ5Bytes, ql::kvq_q5_value);
}

// ------------------------------------------------------------------ q4_0 codec
static void parallel_rows(int64_t rows, int64_t min_rows_per_task,
                          const std::function<void(int64_t, int64_t)>& fn);

int ql_q4_0_pack(const float* w, int64_t rows, int64_t cols, uint16_t* scales,
                 uint8_t* quants) {
    if (!w || !scales || !quants) return set_error(QL_EINVAL, "ql_q4_0_pack: null pointer");
    if (rows <= 0 || cols <= 0 || cols % 32 != 0)
        return set_error(QL_EINVAL, "ql_q4_0_pack: need rows > 0 and cols a positive multiple of 32");
    const int64_t nblk = cols / 32;
    std::vector<int> bad_flags;
    std::mutex mu;
    int bad = 0;
    int64_t bad_row = -1;
    parallel_rows(rows, 64, [&](int64_t r0, int64_t r1) {
        int local = 0;
        int64_t lrow = -1;
        for (int64_t r = r0; r < r1; ++r) {
            for (int64_t j = 0; j < nblk; ++j) {
                int rc = q4_0_block(w + r * cols + j * 32, scales + r * nblk + j,
                                    quants + (r * nblk + j) * 16);
                if (rc && !local) { local = rc; lrow = r; }
            }
        }
        if (local) {
            std::lock_guard<std::mutex> lk(mu);
            if (!bad || lrow < bad_row) { bad = local; bad_row = lrow; }
        }
    });
    if (bad == 1)
        return set_error(QL_EINVAL, "ql_q4_0_pack: non-finite weight in row " + std::to_string(bad_row));
    if (bad == 2)
        return set_error(QL_EINVAL, "ql_q4_0_pack: block scale overflows f16 in row " + std::to_string(bad_row));
    return QL_OK;
}

int ql_q4_0_unpack(const uint16_t* scales, const uint8_t* quants, int64_t rows, int64_t cols,
                   float* w) {
    if (!w || !scales || !quants) return set_error(QL_EINVAL, "ql_q4_0_unpack: null pointer");
    if (rows <= 0 || cols <= 0 || cols % 32 != 0)
        return set_error(QL_EINVAL, "ql_q4_0_unpack: need rows > 0 and cols a positive multiple of 32");
    const int64_t nblk = cols / 32;
    parallel_rows(rows, 64, [&](int64_t r0, int64_t r1) {
        for (int64_t r = r0; r < r1; ++r)
            for (int64_t j = 0; j < nblk; ++j) {
                const double d = f16_to_f64(scales[r * nblk + j]);
                const uint8_t* q = quants + (r * nblk + j) * 16;
                float* o = w + r * cols + j * 32;
                for (int e = 0; e < 16; ++e) {
                    o[e] = (float)(((int)(q[e] & 0xF) - 8) * d);
                    o[e + 16] = (float)(((int)(q[e] >> 4) - 8) * d);
                }
            }
    });
    return QL_OK;
}

int ql_rope_tables(float* h_cos, float* h_sin, int64_t max_position, int head_dim, double theta) {
    if (!h_cos || !h_sin) return set_error(QL_EINVAL, "ql_rope_tables: null pointer");
    if (max_position <= 0 || head_dim <= 0 || head_dim % 2 || !(theta > 0.0))
        return set_error(QL_EINVAL, "ql_rope_tables: bad size or theta");
    const int half = head_dim / 2;
    std::vector<double> inv(half);
    for (int i = 0; i < half; ++i) inv[i] = std::pow(theta, -(2.0 * i) / (double)head_dim);
    parallel_rows(max_position, 256, [&](int64_t p0, int64_t p1) {
        for (int64_t p = p0; p < p1; ++p)
            for (int i = 0; i < half; ++i) {
                const double a = (double)p * inv[i];
                h_cos[p * half + i] = (float)std::cos(a);
                h_sin[p * half + i] = (float)std::sin(a);
            }
    });
    return QL_OK;
}

// ------------------------------------------------------------------ block allocator
struct ql_block_pool {
    int64_t num_blocks = 0;
    int64_t next_id = 0;
    std::vector<int32_t> free_list;   // stack: last freed is reused first
    std::vector<uint8_t> used;
};

int ql_block_pool_create(int64_t num_blocks, ql_block_pool** out) {
    if (!out) return set_error(QL_EINVAL, "ql_block_pool_create: null out");
    if (num_blocks <= 0 || num_blocks > INT32_MAX)
        return set_error(QL_EINVAL, "ql_block_pool_create: num_blocks must be in [1, 2^31)");
    auto* p = new (std::nothrow) ql_block_pool();
    if (!p) return set_error(QL_ENOMEM, "ql_block_pool_create: out of host memory");
    p->num_blocks = num_blocks;
    p->used.assign((size_t)num_blocks, 0);
    *out = p;
    return QL_OK;
}

int ql_block_pool_destroy(ql_block_pool* p) {
    delete p;
    return QL_OK;
}

int ql_block_pool_alloc(ql_block_pool* p, int32_t* out_id) {
    if (!p || !out_id) return set_error(QL_EINVAL, "ql_block_pool_alloc: null pointer");
    int64_t id;
    if (!p->free_list.empty()) {
        id = p->free_list.back();
        p->free_list.pop_back();
    } else if (p->next_id < p->num_blocks) {
        id = p->next_id++;
    } else {
        return set_error(QL_EPOOL, "KV block pool exhausted");
    }
    p->used[(size_t)id] = 1;
    *out_id = (int32_t)id;
    return QL_OK;
}

int ql_block_pool_free(ql_block_pool* p, const int32_t* ids, int64_t n) {
    if (!p || (n > 0 && !ids)) return set_error(QL_EINVAL, "ql_block_pool_free: null pointer");
    for (int64_t i = 0; i < n; ++i) {
        const int64_t id = ids[i];
        if (id < 0 || id >= p->num_blocks || !p->used[(size_t)id])
            return set_error(QL_ERANGE, "ql_block_pool_free: block " + std::to_string(id) +
                                            " is not allocated");
    }
    for (int64_t i = 0; i < n; ++i) {
        p->used[(size_t)ids[i]] = 0;
        p->free_list.push_back(ids[i]);
    }
    return QL_OK;
}

int64_t ql_block_pool_in_use(const ql_block_pool* p) {
    return p ? p->next_id - (int64_t)p->free_list.size() : -1;
}

// ------------------------------------------------------------------ device error record
int ql_check_device_error(ql_model* m) {
    (void)m;
    QL_TRY_CUDA(cudaDeviceSynchronize());
    DevError* d = device_error_record();
    if (!d) return set_error(QL_ECUDA, "ql_check_device_error: no device error record");
    DevError h;
    QL_TRY_CUDA(cudaMemcpy(&h, d, sizeof h, cudaMemcpyDeviceToHost));
    if (!h.code) return QL_OK;
    QL_TRY_CUDA(cudaMemset(d, 0, sizeof h));
    QL_TRY_CUDA(cudaDeviceSynchronize());
    char buf[256];
    std::snprintf(buf, sizeof buf, "%s (index %lld, value %lld)", where_name(h.where), h.index,
                  h.value);
    return set_error(QL_EDEVICE, buf);
}

}  // extern "C"

static void parallel_rows(int64_t rows, int64_t min_rows_per_task,
                          const std::function<void(int64_t, int64_t)>& fn) {
    unsigned hw = std::thread::hardware_concurrency();
    int64_t nt = std::max<int64_t>(1, std::min<int64_t>(hw ? hw : 1, rows / std::max<int64_t>(1, min_rows_per_task)));
    nt = std::min<int64_t>(nt, 64);
    if (nt <= 1) {
        fn(0, rows);
        return;
    }
    std::vector<std::thread> th;
    const int64_t per = (rows + nt - 1) / nt;
    for (int64_t t = 0; t < nt; ++t) {
        const int64_t r0 = t * per, r1 = std::min(rows, r0 + per);
        if (r0 >= r1) break;
        th.emplace_back(fn, r0, r1);
    }
    for (auto& t : th) t.join();
}
