"""The kernels' division by a launch-invariant integer (FastDiv in grouped_gemm.cuh: multiply
by a precomputed reciprocal, Granlund and Montgomery 1994) equals integer division for every
dividend the unit decode can pass (0 <= n < 2^31) and every divisor it uses (tile counts).
Host build of the same header with nvcc; no GPU."""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "moe_ragged_bf16_grouped_b300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <cstdint>
#include <random>
#include "grouped_gemm.cuh"
int main() {
    std::mt19937_64 rng(7);
    long bad = 0, n_checked = 0;
    auto check = [&](uint32_t d, uint32_t n) {
        const gdg::FastDiv f = gdg::FastDiv::make(d);
        ++n_checked;
        if (f.div(n) != n / d) { if (bad < 10) printf("d=%u n=%u got %u\n", d, n, f.div(n)); ++bad; }
    };
    uint32_t ds[] = {1u, 2u, 3u, 5u, 7u, 16u, 28u, 56u, 112u, 255u, 256u, 448u, 1000u, 4096u,
                     65535u, 65536u, 1u << 20, (1u << 30) + 1, 2147483647u};
    for (uint32_t d : ds) {
        for (uint32_t n = 0; n < 70000; ++n) check(d, n);
        for (uint32_t k = 0; k < 20000; ++k) {
            const uint32_t q = static_cast<uint32_t>(rng() % (2147483648ull / d));
            for (int64_t dn = -2; dn <= 2; ++dn) {            // around multiples of d
                const int64_t n = static_cast<int64_t>(q) * d + dn;
                if (n >= 0 && n < 2147483648ll) check(d, static_cast<uint32_t>(n));
            }
            check(d, static_cast<uint32_t>(rng() % 2147483648ull));
        }
        check(d, 2147483647u);
    }
    for (int k = 0; k < 200000; ++k) {                    // random divisors too
        const uint32_t d = 1 + static_cast<uint32_t>(rng() % 2147483647ull);
        check(d, static_cast<uint32_t>(rng() % 2147483648ull));
    }
    printf("checked %ld, bad %ld\n", n_checked, bad);
    return bad != 0;
}
"""


@pytest.mark.skipif(shutil.which("nvcc") is None, reason="needs nvcc")
def test_fastdiv_matches_integer_division():
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "fastdiv.cu")
        with open(src, "w") as f:
            f.write(PROGRAM)
        exe = os.path.join(d, "fastdiv")
        subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17",
                               "-O2", "-I", CSRC, "-o", exe, src])
        r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
        assert r.returncode == 0, r.stdout + r.stderr
        assert "bad 0" in r.stdout
