// Division by a runtime-invariant divisor for 0 <= n < 2^31 (Granlund & Montgomery,
// "Division by invariant integers using multiplication", PLDI 1994):
// q = (mulhi(n, m) + n) >> l with l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1.
#pragma once

#include <cstdint>

namespace pvr {

struct FastDiv {
    uint32_t d, m, l;
};

inline FastDiv make_fastdiv(uint32_t d)
{
    uint32_t l = 0;
    while ((uint64_t(1) << l) < d) ++l;
    const uint64_t m = ((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1;
    return FastDiv{d, static_cast<uint32_t>(m), l};
}

__device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv &f)
{
    return (__umulhi(n, f.m) + n) >> f.l;
}

}  // namespace pvr
