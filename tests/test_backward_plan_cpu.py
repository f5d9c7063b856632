"""Host-side launch plan of the backward's products (csrc/bw_plan.h).

Every product of the backward pass runs as fp32 tiles of 64 x 64 or 128 x 128;
a product with fewer tiles than SMs and a long K is split along K, and the
chunks' partial products are summed in chunk order by a second kernel.  The
plan is host code, compiled here alone, and checked over a sweep of shapes
(the products of the tiny, mid-size and ARMT-1B-shaped cells and ragged
ones) for what the kernels rely on:
  * the chunks cover K exactly once: kchunk is a multiple of 16, ksplit
    chunks of kchunk reach K and ksplit - 1 do not;
  * the partial products fit the scratch the workspace provides;
  * 128 x 128 tiles only when both M and N reach 128 and there is at least one
    tile per SM; splits only for products with fewer tiles than SMs and
    K >= 128, never more chunks than K / 64.
"""
import itertools
import json
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "recurrent_memory_transformer_gb300", "csrc")

PART_CAP = 1 << 22   # the floats of partial-product scratch the backward allocates
SMS = (152, 148, 8)

MS = (1, 16, 20, 64, 80, 127, 128, 528, 1040, 2048, 3072, 16384)
NS = (1, 16, 64, 96, 128, 192, 256, 384, 768, 1024, 2048, 3072, 16384)
KS = (4, 16, 20, 64, 80, 127, 128, 256, 384, 1040, 2048, 8192, 16384)
GS = (1, 2, 4, 16)

PROGRAM = r"""
#include <cstdio>
#include "bw_plan.h"
int main() {
  int M, N, K, G, S; long long cap;
  std::printf("[");
  bool first = true;
  while (std::scanf("%d %d %d %d %d %lld", &M, &N, &K, &G, &S, &cap) == 6) {
    const armt::BwGemmPlan p = armt::bw_gemm_plan(M, N, K, G, S, cap);
    std::printf("%s[%d,%d,%d]", first ? "" : ",", p.bm, p.ksplit, p.kchunk);
    first = false;
  }
  std::printf("]\n");
  return 0;
}
"""


@pytest.fixture(scope="module")
def plans():
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    shapes = [(m, n, k, g, s) for m, n, k, g, s in itertools.product(MS, NS, KS, GS, SMS)]
    with tempfile.TemporaryDirectory() as td:
        src, exe = os.path.join(td, "plan.cpp"), os.path.join(td, "plan")
        open(src, "w").write(PROGRAM)
        r = subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, "-o", exe, src], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
        inp = "\n".join(f"{m} {n} {k} {g} {s} {PART_CAP}" for m, n, k, g, s in shapes)
        out = subprocess.run([exe], input=inp, capture_output=True, text=True, check=True).stdout
    return list(zip(shapes, json.loads(out)))


def test_chunks_cover_k_exactly_once(plans):
    for (m, n, k, g, s), (bm, ks, kc) in plans:
        if ks == 1:
            continue
        assert kc % 16 == 0 and kc > 0, (m, n, k, g, s, kc)
        assert ks * kc >= k and (ks - 1) * kc < k, (m, n, k, g, s, ks, kc)


def test_partials_fit_the_scratch(plans):
    for (m, n, k, g, s), (bm, ks, kc) in plans:
        if ks > 1:
            assert ks * g * m * n <= PART_CAP, (m, n, k, g, s, ks)


def test_tiles_and_splits_only_where_they_apply(plans):
    for (m, n, k, g, s), (bm, ks, kc) in plans:
        assert bm in (64, 128)
        if bm == 128:
            assert m >= 128 and n >= 128
            assert (-(-m // 128)) * (-(-n // 128)) * g >= s
        tiles = (-(-m // bm)) * (-(-n // bm)) * g
        if ks > 1:
            assert tiles < s and k >= 128 and ks <= k // 64, (m, n, k, g, s, ks)
        # the split stays within about two blocks per SM
        assert tiles * ks <= 2 * s + tiles, (m, n, k, g, s, tiles, ks)


def test_plans_of_representative_products(plans):
    # a gate-up-sized product of one ARMT-1B cell fills the GPU with 128 x 128 tiles
    got = {shape: plan for shape, plan in plans}
    assert got[(1040, 16384, 2048, 1, 152)] == [128, 1, 0]
    # [1040 x 8192] x [8192 x 1024] on two cells: 144 tiles of 128 x 128 are fewer than
    # the SMs, so 64 x 64 tiles, enough of them not to split K
    assert got[(1040, 1024, 8192, 2, 152)] == [64, 1, 0]
    # a 16-row memory-row product with a long K is split
    assert got[(16, 384, 2048, 1, 152)][1] > 1
