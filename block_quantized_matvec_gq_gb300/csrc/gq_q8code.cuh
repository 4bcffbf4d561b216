// gq_q8code.cuh -- the Q8_0 code rule for four elements of a 32-block, shared
// by the plain quantizer and the RMS-norm prologue.
//
// "Metal kernel capability table (Phase B ground truth)", section 2
// (quantize_q8): q = clamp(round_half_away(e / d), -127, 127) with d =
// amax / 127 and the division IEEE-rounded; d = 0 gives q = 0.
#pragma once

#include <cstdint>

namespace gq {

// clamp(roundf(e / d), +-127) with the division itself (out of line: rare).
static __device__ __noinline__ int q8_exact_code(float e, float d)
{
    return static_cast<int>(fminf(fmaxf(roundf(__fdiv_rn(e, d)), -127.0f), 127.0f));
}

// The four codes of e (packed, element i in byte i) for the block scale d,
// in full-rate f32 and integer operations only.
//   y = RN(e * RN(1/d)): for |e/d| <= 127, |y - e/d| <= 2^-16 and
//   |RN(e/d) - e/d| <= 2^-17 (relative errors of 2^-24 each), so y and
//   RN(e/d) round to the same integer unless y lies within 2^-15 of a
//   half-integer (or 1/d overflowed).  Those elements take the division
//   itself.
//   Elsewhere no tie is possible, so rounding y to the nearest integer (ties
//   to even or away) gives round_half_away(RN(e/d)).  m = RN(y + 1.5 * 2^23)
//   holds that integer n in its low bits for |y| < 2^22, and y - (m - 1.5 *
//   2^23) = y - n is exact: y lies near a half-integer when |y - n| >=
//   0.5 - 2^-15.
__device__ __forceinline__ uint32_t q8_pack4(const float (&e)[4], float d)
{
    if (d == 0.0f) return 0u;
    constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
    const float r = __frcp_rn(d);
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float y = __fmul_rn(e[i], r);
        const float m = __fadd_rn(y, kMagic);
        const float f = __fsub_rn(y, __fsub_rn(m, kMagic));
        int q;
        if (!(fabsf(y) <= 128.0f) || fabsf(f) >= 0.5f - 0x1p-15f)
            q = q8_exact_code(e[i], d);
        else
            q = __float_as_int(m) - 0x4B400000;
        q = min(max(q, -127), 127);
        packed |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * i);
    }
    return packed;
}

}  // namespace gq
