// Seeded Gumbel noise and the selection key order, shared by the selection
// kernel and the LM-head GEMM's fused selection epilogue.
//
// [COUPLING] (AIexTime post 185): argmax of logits plus Gumbel(0,1) noise is a
// sample from the softmax.  The noise of vocabulary entry v at position p of
// request r is a pure function of (seed, r, p, v): Philox4x32-10 (Salmon et
// al., SC'11) on the counter (v >> 2, p, r, 0) with key (seed lo, seed hi),
// word v & 3, uniform u = (2 (w >> 9) + 1) 2^-24, noise -ln(-ln u) with an fp32
// log made only of correctly rounded IEEE operations.
#pragma once

#include "biv_common.cuh"

namespace biv {

// ----------------------------------------------------------- Philox4x32-10
struct U4 { uint32_t x, y, z, w; };

BIV_DEV U4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
        const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
        const uint32_t n0 = hi1 ^ c1 ^ k0;
        const uint32_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    return U4{c0, c1, c2, c3};
}

// ------------------------------------------------------------- own log
// ln x for positive normal x: x = m 2^e, m in [fl(sqrt2)/2, fl(sqrt2)),
// f = m - 1, s = f / (2 + f), ln m = 2 s sum_{k<=6} s^2k / (2k+1) (Horner,
// fma), ln x = e ln2_hi + (e ln2_lo + ln m), ln2_hi = 0x1.62e4p-1 (17 bits),
// ln2_lo = fl(ln 2 - ln2_hi).  Every step is one correctly rounded IEEE op.
BIV_DEV float own_log(float x) {
    const uint32_t b = __float_as_uint(x);
    int e = static_cast<int>((b >> 23) & 0xffu) - 127;
    const uint32_t frac = b & 0x007fffffu;
    uint32_t mb = frac | 0x3f800000u;
    if (frac >= 0x003504f3u) {
        mb -= 0x00800000u;
        e += 1;
    }
    const float m = __uint_as_float(mb);
    const float f = __fsub_rn(m, 1.0f);
    const float t = __fadd_rn(2.0f, f);
    const float s = __fdiv_rn(f, t);
    const float z = __fmul_rn(s, s);
    float p = __uint_as_float(0x3d9d89d9u);                 // 1/13
    p = __fmaf_rn(p, z, __uint_as_float(0x3dba2e8cu));      // 1/11
    p = __fmaf_rn(p, z, __uint_as_float(0x3de38e39u));      // 1/9
    p = __fmaf_rn(p, z, __uint_as_float(0x3e124925u));      // 1/7
    p = __fmaf_rn(p, z, __uint_as_float(0x3e4ccccdu));      // 1/5
    p = __fmaf_rn(p, z, __uint_as_float(0x3eaaaaabu));      // 1/3
    p = __fmaf_rn(p, z, 1.0f);                              // 1
    const float r = __fadd_rn(s, s);
    const float lnm = __fmul_rn(r, p);
    const float ef = __int2float_rn(e);
    const float u = __fmaf_rn(ef, __uint_as_float(0x35bfbe8eu), lnm);   // ln2_lo
    return __fmaf_rn(ef, __uint_as_float(0x3f317200u), u);              // ln2_hi
}

// u = (2 (w >> 9) + 1) 2^-24 (exact), g = -ln(-ln u).
BIV_DEV float gumbel_from_word(uint32_t w) {
    const float u = __fmul_rn(__uint2float_rn(2u * (w >> 9) + 1u), 5.9604644775390625e-8f);
    const float a = own_log(u);
    return -own_log(-a);
}

// Total order used for selection: NaN lowest, -0 == +0, then by value.
BIV_DEV uint32_t key_order(float k) {
    if (k != k) return 0u;
    if (k == 0.0f) k = 0.0f;
    const uint32_t b = __float_as_uint(k);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

BIV_DEV unsigned long long pack_key(float k, uint32_t v) {
    return (static_cast<unsigned long long>(key_order(k)) << 32) | static_cast<unsigned long long>(~v);
}

BIV_DEV unsigned long long umax64(unsigned long long a, unsigned long long b) { return a > b ? a : b; }

BIV_DEV unsigned long long warp_max64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = umax64(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}


}  // namespace biv
