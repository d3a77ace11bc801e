// pack.cpp -- the fixed-stride expert blob (layout v1, see moe.h) and its packer.
//
// The Swiftlet pages fix only that every routed expert is one fixed-stride blob
// so that one read fetches one expert (article section 2 "Fixed-stride pread
// reads"; README "How it works").  Sections, bit order and padding are this
// library's layout: codes low bits first, eight 4-bit (or four 8-bit) codes
// per little-endian 32-bit word, fp16 (scale, bias) per 64-column group, and
// the stride rounded up to 4096 bytes so every blob starts page aligned.
#include <cstring>

#include "moe_internal.h"

namespace {

bool valid_shape(int32_t hidden, int32_t inter, int32_t bits) {
    return (bits == 4 || bits == 8) && hidden > 0 && inter > 0 && hidden % 64 == 0 && inter % 64 == 0;
}

uint8_t* put_codes(uint8_t* dst, const uint8_t* q, int32_t rows, int32_t cols, int32_t bits) {
    const int per = 32 / bits;
    for (int64_t r = 0; r < rows; ++r) {
        const uint8_t* row = q + r * cols;
        for (int32_t c = 0; c < cols; c += per) {
            uint32_t v = 0;
            for (int i = 0; i < per; ++i) v |= (uint32_t)row[c + i] << (i * bits);
            dst[0] = (uint8_t)v;
            dst[1] = (uint8_t)(v >> 8);
            dst[2] = (uint8_t)(v >> 16);
            dst[3] = (uint8_t)(v >> 24);
            dst += 4;
        }
    }
    return dst;
}

uint8_t* put_scale_bias(uint8_t* dst, const uint16_t* sb, int32_t rows, int32_t cols) {
    const int64_t n = (int64_t)rows * (cols / 64);
    for (int64_t g = 0; g < n; ++g) {
        const uint16_t s = sb[2 * g], b = sb[2 * g + 1];
        dst[0] = (uint8_t)s;
        dst[1] = (uint8_t)(s >> 8);
        dst[2] = (uint8_t)b;
        dst[3] = (uint8_t)(b >> 8);
        dst += 4;
    }
    return dst;
}

bool codes_in_range(const uint8_t* q, int64_t n, int32_t bits) {
    const uint8_t lim = (uint8_t)((1u << bits) - 1u);
    for (int64_t i = 0; i < n; ++i)
        if (q[i] > lim) return false;
    return true;
}

}  // namespace

extern "C" size_t moe_blob_bytes(int32_t hidden, int32_t inter, int32_t bits) {
    if (!valid_shape(hidden, inter, bits)) return 0;
    return (size_t)moe::blob_layout(hidden, inter, bits).bytes;
}

extern "C" size_t moe_blob_stride(int32_t hidden, int32_t inter, int32_t bits) {
    const size_t b = moe_blob_bytes(hidden, inter, bits);
    return (b + 4095) / 4096 * 4096;
}

extern "C" int moe_pack_expert(int32_t hidden, int32_t inter, int32_t bits, const uint8_t* q_gate,
                               const uint16_t* sb_gate, const uint8_t* q_up, const uint16_t* sb_up,
                               const uint8_t* q_down, const uint16_t* sb_down, void* blob, size_t blob_bytes) {
    if (!valid_shape(hidden, inter, bits) || !q_gate || !sb_gate || !q_up || !sb_up || !q_down || !sb_down ||
        !blob)
        return MOE_EINVAL;
    const size_t stride = moe_blob_stride(hidden, inter, bits);
    if (blob_bytes < stride) return MOE_EINVAL;
    const int64_t n = (int64_t)hidden * inter;
    if (!codes_in_range(q_gate, n, bits) || !codes_in_range(q_up, n, bits) || !codes_in_range(q_down, n, bits))
        return MOE_EINVAL;
    uint8_t* p = static_cast<uint8_t*>(blob);
    std::memset(p, 0, stride);
    p = put_codes(p, q_gate, inter, hidden, bits);
    p = put_codes(p, q_up, inter, hidden, bits);
    p = put_codes(p, q_down, hidden, inter, bits);
    p = put_scale_bias(p, sb_gate, inter, hidden);
    p = put_scale_bias(p, sb_up, inter, hidden);
    put_scale_bias(p, sb_down, hidden, inter);
    return MOE_OK;
}
