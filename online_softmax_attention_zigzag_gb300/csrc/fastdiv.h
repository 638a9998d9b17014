// fastdiv.h -- division of n < 2^31 by a fixed d >= 1 with one wide multiply and a shift
// (Granlund and Montgomery, "Division by invariant integers using multiplication", 1994):
// with l = ceil(log2 d) and mult = ceil(2^(31+l) / d), n / d = (n * mult) >> (31+l)
// exactly, because n * (mult - 2^(31+l)/d) / 2^(31+l) < 2^-l <= 1/d.
// Plain C++ when compiled by a host compiler, so the host can check it.
#pragma once

#ifdef __CUDACC__
#define RA_HD __host__ __device__ __forceinline__
#else
#define RA_HD inline
#endif

namespace ra {

struct FastDiv {
    unsigned long long mult;
    int shift;
    unsigned d;
};

inline FastDiv make_fastdiv(unsigned d) {
    int l = 0;
    while ((1ull << l) < d) ++l;
    const unsigned long long num = 1ull << (31 + l);
    FastDiv f;
    f.mult = (num + d - 1) / d;
    f.shift = 31 + l;
    f.d = d;
    return f;
}

RA_HD unsigned fdiv(unsigned n, const FastDiv& f) {
    return static_cast<unsigned>((static_cast<unsigned long long>(n) * f.mult) >> f.shift);
}

}  // namespace ra
