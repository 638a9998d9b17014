"""The relayout kernel's division by invariant integers (csrc/fastdiv.h), host-compiled
with g++ and checked against integer division (CPU only).

Granlund and Montgomery's bound makes (n * mult) >> shift equal n / d for every n < 2^31;
the harness checks that claim for every divisor up to 300 and a sample of divisors up to
10^6, each against a set of numerators that includes 0, the multiples of d and their
neighbours, the largest n < 2^31 and random values.
"""
import os
import shutil
import subprocess

import pytest

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "online_softmax_attention_zigzag_gb300", "csrc")

HARNESS = r"""
#include <cstdio>
#include <cstdint>
#include <random>
#include "fastdiv.h"

static int check(unsigned d, std::mt19937_64& rng) {
    const ra::FastDiv f = ra::make_fastdiv(d);
    const unsigned top = 0x7fffffffu;
    auto one = [&](unsigned n) -> int {
        if (ra::fdiv(n, f) != n / d) { std::printf("fail d=%u n=%u\n", d, n); return 1; }
        return 0;
    };
    int bad = 0;
    for (unsigned n = 0; n < 4096u; ++n) bad += one(n);
    for (unsigned k = 1; k < 2000u; ++k) {
        const unsigned long long m = static_cast<unsigned long long>(d) * k;
        if (m + 1 > top) break;
        bad += one(static_cast<unsigned>(m - 1)) + one(static_cast<unsigned>(m)) + one(static_cast<unsigned>(m + 1));
    }
    const unsigned q = top / d;  // multiples near the top of the range
    for (unsigned k = (q > 4 ? q - 4 : 0); k <= q; ++k) {
        const unsigned long long m = static_cast<unsigned long long>(d) * k;
        if (m <= top) bad += one(static_cast<unsigned>(m));
        if (m >= 1 && m - 1 <= top) bad += one(static_cast<unsigned>(m - 1));
    }
    bad += one(top) + one(top - 1);
    for (int i = 0; i < 20000; ++i) bad += one(static_cast<unsigned>(rng() & top));
    return bad;
}

int main() {
    std::mt19937_64 rng(12345);
    int bad = 0;
    for (unsigned d = 1; d <= 300u; ++d) bad += check(d, rng);
    for (int i = 0; i < 300; ++i) bad += check(301u + static_cast<unsigned>(rng() % 999700u), rng);
    bad += check(1000000u, rng);
    std::printf(bad ? "FAILED %d\n" : "ok\n", bad);
    return bad ? 1 : 0;
}
"""


def test_fastdiv_matches_integer_division(tmp_path):
    gxx = shutil.which("g++") or shutil.which("c++")
    if gxx is None:
        pytest.skip("no host C++ compiler")
    src = tmp_path / "fastdiv_check.cpp"
    src.write_text(HARNESS)
    exe = tmp_path / "fastdiv_check"
    subprocess.run([gxx, "-O2", "-std=c++17", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], stdout=subprocess.PIPE, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout[-2000:]
