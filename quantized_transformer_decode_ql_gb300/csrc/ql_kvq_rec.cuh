// The quantised KV pool of the attention: keys as q8_0 rows, values as q5_1 rows.
//
// memra-engine qwen4exp_gpu.rs, the quantised-cache storage (the Q8Q5 store, q8_row_bytes /
// q5_row_bytes) and its host twins host_quant_q8_row / host_quant_q5_row: a row is cut into
// 32-element blocks; q8_0 keeps an f16 scale d = max|x| / 127 and 32 codes round(x / d) in
// [-127, 127]; q5_1 keeps an f16 scale d = (max - min) / 31, an f16 minimum m and 32 codes
// round((x - min) / d) in [0, 31] (low four bits as nibbles, bit 4 in a 32-bit word). Every step
// is one f32 operation; the f16 conversions round to nearest even.
//
// Layout (GB300): one record per (physical block, kv head) of a layer, holding the block's 16 key
// rows and 16 value rows with each field in its own array, so that the record is one contiguous
// run of 29 * head_dim bytes whose fields all start on 16-byte boundaries (the page's interleaved
// 34- and 24-byte blocks would not): a tile of the cache is one copy, 3712 bytes at head_dim 128
// against 8192 for f16 K and V.
//   KC  int8 [16][HD]        key codes               at 0
//   VN  u8   [16][HD / 2]    value nibbles (per block: byte l = code l | code l+16 << 4) at 16 HD
//   KD  f16  [16][HD / 32]   key scales              at 24 HD
//   VH  u32  [16][HD / 32]   value bit 4 (bit l = code l's) at 25 HD
//   VD  f16  [16][HD / 32]   value scales            at 27 HD
//   VM  f16  [16][HD / 32]   value minima            at 28 HD
// A block's bytes in the page's format are KD, KC[32 b .. 32 b + 31] (q8_0) and VD, VM, VH,
// VN[16 b .. 16 b + 15] (q5_1): the same values, only the order differs.
#pragma once

#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

#include "ql_internal.h"

namespace ql {

template <int HD>
struct Kvq {
    static constexpr int NB = HD / 32;   // 32-element blocks per row
    static constexpr int KC = 0, VN = 16 * HD, KD = 24 * HD, VH = 25 * HD, VD = 27 * HD, VM = 28 * HD;
    static constexpr int BYTES = 29 * HD;
};

#ifdef __CUDACC__
__device__ __forceinline__ float kvq_inv(float d) {
    if (d == 0.0f) return 0.0f;
    const float id = __fdiv_rn(1.0f, d);
    return isfinite(id) ? id : 0.0f;
}

// Quantise one key row into slot `slot` of a record, by one warp: x[k] is element lane of block k
// (dimension lane + 32 k). Writes the codes and scales; dec (shared memory, optional) receives
// the decoded f16 row as the attention reads it back (f16(d * code)). Returns false (every lane)
// if a scale overflowed f16.
template <int HD>
__device__ __forceinline__ bool kvq_put_k_row(const float (&x)[HD / 32], uint8_t* rec, int slot, int lane,
                                              __half* dec) {
    bool ok = true;
#pragma unroll
    for (int k = 0; k < Kvq<HD>::NB; ++k) {
        float a = fabsf(x[k]);
#pragma unroll
        for (int o = 16; o; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        const float d = __fdiv_rn(a, 127.0f);
        const float id = kvq_inv(d);
        float qf = rintf(__fmul_rn(x[k], id));
        qf = fminf(fmaxf(qf, -127.0f), 127.0f);
        const int q = (int)qf;
        rec[Kvq<HD>::KC + slot * HD + 32 * k + lane] = (uint8_t)(int8_t)q;
        const __half dh = __float2half_rn(d);
        if (lane == 0) reinterpret_cast<__half*>(rec + Kvq<HD>::KD)[slot * Kvq<HD>::NB + k] = dh;
        ok = ok && !__hisinf(dh);
        if (dec != nullptr) dec[32 * k + lane] = __hmul(__int2half_rn(q), dh);
    }
    return ok;
}

// The same for one value row as q5_1 (dec: f16(fma(d, code, m)), as the attention decodes it).
template <int HD>
__device__ __forceinline__ bool kvq_put_v_row(const float (&x)[HD / 32], uint8_t* rec, int slot, int lane,
                                              __half* dec) {
    bool ok = true;
#pragma unroll
    for (int k = 0; k < Kvq<HD>::NB; ++k) {
        float mn = x[k], mx = x[k];
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
        mn = __fadd_rn(mn, 0.0f);   // a zero minimum is stored as +0
        const float d = __fdiv_rn(__fsub_rn(mx, mn), 31.0f);
        const float id = kvq_inv(d);
        float qf = rintf(__fmul_rn(__fsub_rn(x[k], mn), id));
        qf = fminf(fmaxf(qf, 0.0f), 31.0f);
        const uint32_t c = (uint32_t)qf;
        const uint32_t qh = __ballot_sync(0xffffffffu, (c >> 4) & 1u);
        const uint32_t c16 = __shfl_down_sync(0xffffffffu, c, 16);
        if (lane < 16) rec[Kvq<HD>::VN + slot * (HD / 2) + 16 * k + lane] = (uint8_t)((c & 0xFu) | ((c16 & 0xFu) << 4));
        const __half dh = __float2half_rn(d), mh = __float2half_rn(mn);
        if (lane == 0) {
            reinterpret_cast<uint32_t*>(rec + Kvq<HD>::VH)[slot * Kvq<HD>::NB + k] = qh;
            reinterpret_cast<__half*>(rec + Kvq<HD>::VD)[slot * Kvq<HD>::NB + k] = dh;
            reinterpret_cast<__half*>(rec + Kvq<HD>::VM)[slot * Kvq<HD>::NB + k] = mh;
        }
        ok = ok && !__hisinf(dh) && !__hisinf(mh);
        if (dec != nullptr) dec[32 * k + lane] = __hfma(__uint2half_rn(c), dh, mh);
    }
    return ok;
}

// Decode a record staged in shared memory into f16 key and value tiles [16][HD] (row pitch
// `pitch` bytes), by one warp: keys f16(d * code) (HMUL2 of the exact f16 code), values
// f16(fma(d, code, m)) (HFMA2). Codes become exact f16 through the exponent of 1024.
template <int HD>
__device__ __forceinline__ void kvq_decode_tile(const unsigned char* rec, unsigned char* ktile, unsigned char* vtile,
                                                int pitch, int lane) {
    constexpr int CH = HD / 8;   // 8-element chunks per row
    const __half2 k1152 = __float2half2_rn(1152.0f), k1024 = __float2half2_rn(1024.0f);
    auto h2 = [](uint32_t u) {
        __half2 h;
        *reinterpret_cast<uint32_t*>(&h) = u;
        return h;
    };
    auto u32 = [](__half2 h) { return *reinterpret_cast<uint32_t*>(&h); };
    for (int c = lane; c < 16 * CH; c += 32) {
        const int row = c / CH, cc = c - row * CH, blk = cc >> 2;
        // keys: 8 signed codes; (byte ^ 0x80) | 0x6400 is 1152 + code exactly
        const uint2 kc = *reinterpret_cast<const uint2*>(rec + Kvq<HD>::KC + row * HD + 8 * cc);
        const __half d = reinterpret_cast<const __half*>(rec + Kvq<HD>::KD)[row * Kvq<HD>::NB + blk];
        const __half2 dd = __half2half2(d);
        const uint32_t a = kc.x ^ 0x80808080u, b = kc.y ^ 0x80808080u;
        uint4 ko;
        ko.x = u32(__hmul2(__hsub2(h2(__byte_perm(a, 0x64646464u, 0x5140)), k1152), dd));
        ko.y = u32(__hmul2(__hsub2(h2(__byte_perm(a, 0x64646464u, 0x7362)), k1152), dd));
        ko.z = u32(__hmul2(__hsub2(h2(__byte_perm(b, 0x64646464u, 0x5140)), k1152), dd));
        ko.w = u32(__hmul2(__hsub2(h2(__byte_perm(b, 0x64646464u, 0x7362)), k1152), dd));
        *reinterpret_cast<uint4*>(ktile + row * pitch + cc * 16) = ko;
        // values: elements l..l+7 of block blk (l = 8 (cc & 3)); low nibbles of bytes l..l+7 for
        // l < 16, else high nibbles of bytes l-16..l-9; bit 4 from the block's word
        const int l = 8 * (cc & 3);
        const uint2 vb = *reinterpret_cast<const uint2*>(rec + Kvq<HD>::VN + row * (HD / 2) + 16 * blk + (l & 15));
        const uint32_t sh = l < 16 ? 0u : 4u;
        const uint32_t qh = reinterpret_cast<const uint32_t*>(rec + Kvq<HD>::VH)[row * Kvq<HD>::NB + blk] >> l;
        // bit j of t lands in bit 4 of byte j (the multiplier's shifted copies do not overlap)
        const uint32_t t0 = qh & 0xFu, t1 = (qh >> 4) & 0xFu;
        const uint32_t c0 = ((vb.x >> sh) & 0x0F0F0F0Fu) | (((t0 * 0x00204081u) & 0x01010101u) << 4);
        const uint32_t c1 = ((vb.y >> sh) & 0x0F0F0F0Fu) | (((t1 * 0x00204081u) & 0x01010101u) << 4);
        const __half2 vd = __half2half2(reinterpret_cast<const __half*>(rec + Kvq<HD>::VD)[row * Kvq<HD>::NB + blk]);
        const __half2 vm = __half2half2(reinterpret_cast<const __half*>(rec + Kvq<HD>::VM)[row * Kvq<HD>::NB + blk]);
        uint4 vo;
        vo.x = u32(__hfma2(__hsub2(h2(__byte_perm(c0, 0x64646464u, 0x5140)), k1024), vd, vm));
        vo.y = u32(__hfma2(__hsub2(h2(__byte_perm(c0, 0x64646464u, 0x7362)), k1024), vd, vm));
        vo.z = u32(__hfma2(__hsub2(h2(__byte_perm(c1, 0x64646464u, 0x5140)), k1024), vd, vm));
        vo.w = u32(__hfma2(__hsub2(h2(__byte_perm(c1, 0x64646464u, 0x7362)), k1024), vd, vm));
        *reinterpret_cast<uint4*>(vtile + row * pitch + cc * 16) = vo;
    }
}
#endif

}  // namespace ql
