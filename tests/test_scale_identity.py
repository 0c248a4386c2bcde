"""The GPU quantizers compute the Q8_0 block scale amax / 127 without a division:
q = fl(amax * C) with C = fl(1/127), r = fma(-q, 127, amax), d = fma(r, C, q).
This CPU test checks that identity against IEEE division on a strided sample of
every positive finite binary32 (all exponents and mantissa phases), plus the
Q4_0 scale amax / 8 == amax * 0.125.  Set Q4Q_EXHAUSTIVE=1 to check all 2^31 - 2^23
positive finite patterns (about 30 s on 8 cores).
"""
import os
import subprocess

SRC = r"""
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>
#include <stdlib.h>
static float bf(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
int main(int argc, char** argv) {
    const int64_t stride = atoll(argv[1]);
    const float C = 1.0f / 127.0f;
    unsigned long long bad = 0, n = 0;
    #pragma omp parallel for reduction(+:bad, n) schedule(static)
    for (int64_t u = 1; u < 0x7f800000LL; u += stride) {
        float a = bf((uint32_t)u);
        float q = a * C;
        float r = fmaf(-q, 127.0f, a);
        float d = fmaf(r, C, q);
        if (d != a / 127.0f) bad++;
        if (a * 0.125f != a / 8.0f) bad++;
        n++;
    }
    printf("%llu %llu\n", n, bad);
    return 0;
}
"""


def test_division_free_block_scales(tmp_path):
    c = tmp_path / "scale.c"
    exe = tmp_path / "scale"
    c.write_text(SRC)
    subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-o", str(exe), str(c), "-lm"], check=True)
    stride = "1" if os.environ.get("Q4Q_EXHAUSTIVE") == "1" else "61"
    out = subprocess.run([str(exe), stride], capture_output=True, text=True, check=True).stdout.split()
    n, bad = int(out[0]), int(out[1])
    assert n > 30_000_000 and bad == 0
