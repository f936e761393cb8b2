"""Host logic of the tensor-core kernels' work split (the 32-bit helpers the
kernels evaluate in their prologue and epilogue, from the library's internal
header): for many (tiles, stages per tile, clusters, cluster size) every stage
of every tile belongs to exactly one rank, the ranks' ranges are contiguous and
ascending, and the rank that holds a stage is the one rank_of names.  Compiled
with the host C++ compiler; no GPU."""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SRC = r'''
#include <cstdio>
#include <vector>
#include "lbq_internal.h"
int main() {
    long long checked = 0;
    const int Ts[] = {1, 2, 3, 5, 16, 32, 56, 79, 112, 140, 313, 1002};
    const int Uts[] = {4, 8, 12, 16, 56, 67, 232, 1152};
    for (int T : Ts)
        for (int Ut : Uts)
            for (int C = 1; C <= 16; ++C)
                for (int G : {1, 2, 7, 28, 38, 152}) {
                    if (G > T) continue;
                    if ((long long)T * Ut * 16 >= (1ll << 31)) continue;
                    std::vector<int> owner((size_t)T * Ut, -1);
                    for (int cl = 0; cl < G; ++cl) {
                        int t0, t1;
                        lbq::cluster_tiles(T, G, cl, &t0, &t1);
                        if (t0 < 0 || t1 > T || t1 < t0) { printf("bad tiles\n"); return 1; }
                        const int units = (t1 - t0) * Ut;
                        int prev = 0;
                        for (int r = 0; r < C; ++r) {
                            int u0, u1;
                            lbq::rank_range(units, C, r, &u0, &u1);
                            if (u0 != prev || u1 < u0) { printf("not contiguous\n"); return 1; }
                            prev = u1;
                            for (int u = u0; u < u1; ++u) {
                                const size_t g = (size_t)t0 * Ut + u;
                                if (owner[g] != -1) { printf("stage twice\n"); return 1; }
                                owner[g] = cl * C + r;
                                if (lbq::rank_of(units, C, u) != r) { printf("rank_of %d %d %d\n", units, C, u); return 1; }
                                ++checked;
                            }
                        }
                        if (prev != units) { printf("ranges short\n"); return 1; }
                    }
                    for (int o : owner)
                        if (o < 0) { printf("stage missed\n"); return 1; }
                }
    printf("ok %lld\n", checked);
    return 0;
}
'''


def test_work_split_covers_every_stage_once():
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "split.cpp")
        exe = os.path.join(d, "split")
        with open(src, "w") as f:
            f.write(SRC)
        subprocess.run([cxx, "-std=c++17", "-O1", "-I" + os.path.join(ROOT, "include"),
                        "-I" + os.path.join(ROOT, "bit_weight_only_lbq_gb300", "csrc"), src, "-o", exe],
                       check=True, capture_output=True)
        out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
        assert out.returncode == 0, out.stdout + out.stderr
        assert out.stdout.startswith("ok ")
