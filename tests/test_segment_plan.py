"""Host-side pins of the segmented walk's planning (no GPU): the cost model's choices on the
pages' workloads and the balanced cut of the chained form, compiled from the library's own
header as host code and checked against an independent greedy cut written here."""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "linear_attention_serving_02_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "kda_common.cuh"
int main() {
    const long long shapes[][3] = {{1 << 20, 1, 12}, {8192, 1, 12}, {117560, 8, 32}, {30720, 3, 5}, {8192, 1, 4}};
    for (auto &x : shapes) {
        const kda::SegShape r = kda::walk_segments(x[0], x[1], x[2]);
        printf("shape %lld %lld %lld %d %d %d\n", x[0], x[1], x[2], r.P, r.E,
               (int)kda::walk_chain_mode(x[0], x[1], x[2]));
    }
    // the balanced cut as the plan kernel applies it: segment k takes len_at(level, k),
    // less one if it grew at that level and is among the last `surplus` segments that did
    int len_p[][2] = {{128, 19}, {39, 19}, {21, 10}, {157, 10}, {47, 5}, {1000, 37}, {5000, 201}, {64, 4}};
    for (auto &lp : len_p) {
        const int len = lp[0], P = lp[1], S = (len + P - 1) / P;
        const kda::BalancedCut cut(len, P, S);
        printf("cut %d %d", len, P);
        int seen = 0;
        for (int k = 0; k < S; ++k) {
            int L = kda::BalancedCut::len_at(cut.level, k, P);
            if (cut.grew(k)) {
                if (seen >= cut.grown - cut.surplus) --L;
                ++seen;
            }
            printf(" %d", L);
        }
        printf(" last %d\n", cut.last_len());
    }
    return 0;
}
"""


def _run():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    d = tempfile.mkdtemp()
    src, exe = os.path.join(d, "plan.cu"), os.path.join(d, "plan")
    open(src, "w").write(PROGRAM)
    subprocess.check_call([nvcc, "-std=c++17", "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"),
                           "-I", CSRC, src, "-o", exe])
    out = subprocess.check_output([exe], text=True)
    shutil.rmtree(d, ignore_errors=True)
    return out


def _greedy_cut(length, P, step16=9):
    """Start every segment at P chunks and take the surplus back one chunk at a time from
    the segment whose chain plus chunks (16 L + step16 (k - 1), in 1/16 chunk steps) is
    largest, the later one on a tie: the cut that evens out the output walks' critical paths."""
    S = -(-length // P)
    L = [P] * S
    for _ in range(S * P - length):
        cost = [16 * L[k] + step16 * max(k - 1, 0) if L[k] > 1 else -1 for k in range(S)]
        k = max(range(S), key=lambda i: (cost[i], i))
        L[k] -= 1
    return L


@pytest.fixture(scope="module")
def plan_output():
    return _run()


def test_cost_model_choices(plan_output):
    shapes = {}
    for line in plan_output.splitlines():
        if line.startswith("shape"):
            t, n, h, P, E, chain = map(int, line.split()[1:])
            shapes[(t, n, h)] = (P, E, chain)
    assert shapes[(1 << 20, 1, 12)] == (328, 4, 0)   # combine form, long end segments
    assert shapes[(8192, 1, 12)] == (19, 1, 1)       # chained form, 7 segments
    assert shapes[(117560, 8, 32)] == (0, 1, 0)      # 256 chains fill the GPU: plain walk
    assert shapes[(30720, 3, 5)] == (16, 1, 0)       # combine form, uniform
    assert shapes[(8192, 1, 4)][2] == 1


def test_balanced_cut_matches_the_greedy_cut(plan_output):
    n = 0
    for line in plan_output.splitlines():
        if not line.startswith("cut"):
            continue
        f = line.split()
        length, P = int(f[1]), int(f[2])
        i = f.index("last")
        L = list(map(int, f[3:i]))
        assert sum(L) == length and all(1 <= x <= P for x in L), line
        assert L[-1] == int(f[i + 1]), line  # the host's last-segment length (the deferral uses it)
        g = _greedy_cut(length, P)
        cost = lambda c: max(16 * c[k] + 9 * max(k - 1, 0) for k in range(len(c)))
        assert cost(L) == cost(g), (line, g)  # the same critical path
        n += 1
    assert n == 8
    assert _greedy_cut(128, 19) == [19, 19, 19, 19, 18, 17, 17]
