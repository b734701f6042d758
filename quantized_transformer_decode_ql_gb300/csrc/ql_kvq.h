// Quantised KV-cache rows: q8_0 (keys) and q5_1 (values), usable from host and device code.
//
// memra-engine qwen4exp_gpu.rs, the quantised-cache storage (q8_row_bytes / q5_row_bytes,
// the Q8Q5 store) and its host twins (host_quant_q8_row, host_deq_q8_rows, host_quant_q5_row,
// host_deq_q5_rows), which the page keeps bit-identical to its device kernels. Every step is
// an f32 operation; the f16 conversions round to nearest, ties to even. A row is cut into
// 32-element blocks; a ragged last block is padded with zeros, which take part in its
// statistics.
//
// q8_0, 34 bytes per block: f16 d (little-endian), 32 signed 8-bit codes.
//   amax = max |x|, d = amax / 127, id = 1 / d (0 if d == 0 or 1 / d is not finite),
//   code = clamp(rint(x * id), -127, 127). Decoded: f32(d16) * code (exact).
// q5_1, 24 bytes per block: f16 d, f16 m, a 32-bit word (bit l = bit 4 of code l), 16 bytes
//   (byte l: code l's low four bits, then code l + 16's in the high nibble).
//   d = (max - min) / 31, id as above, code = clamp(rint((x - min) * id), 0, 31), m = min.
//   Decoded: fma(f32(d16), code, f32(m16)); d16 * code is exact, so this is one f32 rounding.
#pragma once

#include <stdint.h>
#include <math.h>

#include "ql_f16.h"

namespace ql {

constexpr int kKvqBlock = 32, kQ8Bytes = 34, kQ5Bytes = 24;

QL_HD float kvq_at(const float* x, int n, int l) { return l < n ? x[l] : 0.0f; }

QL_HD float kvq_inverse(float d) {
    if (d == 0.0f) return 0.0f;
    const float id = 1.0f / d;
    return isfinite(id) ? id : 0.0f;
}

// One q8_0 block from x[0..n) (n <= 32, the rest zeros). Returns 0, or 2 if the scale
// overflows f16.
QL_HD int kvq_q8_block(const float* x, int n, uint8_t* out) {
    float amax = 0.0f;
    for (int l = 0; l < kKvqBlock; ++l) amax = fmaxf(amax, fabsf(kvq_at(x, n, l)));
    const float d = amax / 127.0f;
    const float id = kvq_inverse(d);
    const uint16_t dh = f64_to_f16_rne((double)d);
    out[0] = (uint8_t)(dh & 0xFF);
    out[1] = (uint8_t)(dh >> 8);
    for (int l = 0; l < kKvqBlock; ++l) {
        float q = rintf(kvq_at(x, n, l) * id);
        q = fminf(fmaxf(q, -127.0f), 127.0f);
        out[2 + l] = (uint8_t)(int8_t)(int)q;
    }
    return (dh & 0x7C00u) == 0x7C00u ? 2 : 0;
}

QL_HD float kvq_q8_value(const uint8_t* blk, int l) {
    const float d = (float)f16_to_f64((uint16_t)(blk[0] | (blk[1] << 8)));
    return d * (float)(int8_t)blk[2 + l];
}

// One q5_1 block from x[0..n) (n <= 32, the rest zeros). Returns 0, or 2 if d or m overflows
// f16.
QL_HD int kvq_q5_block(const float* x, int n, uint8_t* out) {
    float mn = INFINITY, mx = -INFINITY;
    for (int l = 0; l < kKvqBlock; ++l) {
        const float v = kvq_at(x, n, l);
        mn = fminf(mn, v);
        mx = fmaxf(mx, v);
    }
    mn += 0.0f;   // a zero minimum (-0 or +0: the page does not say which) is stored as +0
    const float d = (mx - mn) / 31.0f;
    const float id = kvq_inverse(d);
    uint32_t qh = 0;
    uint8_t lo[kKvqBlock];
    for (int l = 0; l < kKvqBlock; ++l) {
        float q = rintf((kvq_at(x, n, l) - mn) * id);
        q = fminf(fmaxf(q, 0.0f), 31.0f);
        const uint32_t c = (uint32_t)q;
        qh |= ((c >> 4) & 1u) << l;
        lo[l] = (uint8_t)(c & 0x0Fu);
    }
    const uint16_t dh = f64_to_f16_rne((double)d), mh = f64_to_f16_rne((double)mn);
    out[0] = (uint8_t)(dh & 0xFF);
    out[1] = (uint8_t)(dh >> 8);
    out[2] = (uint8_t)(mh & 0xFF);
    out[3] = (uint8_t)(mh >> 8);
    for (int k = 0; k < 4; ++k) out[4 + k] = (uint8_t)(qh >> (8 * k));
    for (int l = 0; l < 16; ++l) out[8 + l] = (uint8_t)(lo[l] | (lo[l + 16] << 4));
    return ((dh & 0x7C00u) == 0x7C00u || (mh & 0x7C00u) == 0x7C00u) ? 2 : 0;
}

QL_HD float kvq_q5_value(const uint8_t* blk, int l) {
    const float d = (float)f16_to_f64((uint16_t)(blk[0] | (blk[1] << 8)));
    const float m = (float)f16_to_f64((uint16_t)(blk[2] | (blk[3] << 8)));
    const uint32_t qh = (uint32_t)blk[4] | ((uint32_t)blk[5] << 8) | ((uint32_t)blk[6] << 16) |
                        ((uint32_t)blk[7] << 24);
    const uint32_t nib = l < 16 ? (blk[8 + l] & 0x0Fu) : (blk[8 + l - 16] >> 4);
    const uint32_t c = nib | (((qh >> l) & 1u) << 4);
    return fmaf(d, (float)c, m);
}

}  // namespace ql
