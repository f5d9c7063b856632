"""Host-side schedule arithmetic of the library (csrc/schedule.h), compiled
alone with the host C++ compiler and checked against properties of the
layer x segment grid: the summary page (section 二) fixes that cell (l, s)
needs (l-1, s) and (l, s-1), that step i holds the cells with l + s = i, and
that L + n - 1 steps cover the grid.  Also the bookkeeping of results that
are final after a step (used to copy them to the host while the forward
runs), the cell of a short last segment, and the pair-tile rule."""
import json
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "recurrent_memory_transformer_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <initializer_list>
#include "schedule.h"
using namespace armt;
int main() {
  const int Ls[] = {1, 2, 3, 16};
  const long long ns[] = {1, 2, 5, 17};
  const int S = 16;
  std::printf("[");
  bool first = true;
  for (int L : Ls)
    for (long long n : ns)
      for (int cut : {0, 1, 15}) {
        const long long n_tok = n * S - (n * S > cut ? cut : 0);
        const long long n2 = n_segments_for(n_tok, S);
        std::printf("%s{\"L\":%d,\"n\":%lld,\"S\":%d,\"n_tok\":%lld,\"n_seg\":%lld,\"last_len\":%d,\"steps\":[",
                    first ? "" : ",", L, n, S, n_tok, n2, last_segment_len(n_tok, S));
        first = false;
        for (long long i = 0; i < diagonal_steps(L, n2); ++i) {
          CellRange c = diagonal_step(i, L, n2);
          std::printf("%s[%d,%d,%lld,%lld,%lld,%d]", i ? "," : "", c.lo, c.hi, c.s_lo,
                      last_segment_layer(c.lo, c.s_lo, n2), diagonal_rows_final(i, L, S, n_tok),
                      diagonal_layers_final(i, n2));
        }
        std::printf("],\"seq\":[");
        for (long long s = 0; s < n2; ++s)
          std::printf("%s[%lld,%d]", s ? "," : "", sequential_rows_final(s, S, n_tok),
                      sequential_layers_final(s, n2, L));
        std::printf("]}");
      }
  std::printf("]\n");
  std::printf("{");
  const long long rows[] = {16, 128, 200, 256, 300, 1040, 2080, 4160, 8192, 8320, 16640, 131072};
  for (int k = 0; k < 12; ++k) std::printf("%s\"%lld\":%d", k ? "," : "", rows[k], pair_tiles_pay_off(rows[k]) ? 1 : 0);
  std::printf("}\n");
  return 0;
}
"""


@pytest.fixture(scope="module")
def output():
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    d = tempfile.mkdtemp()
    src, exe = os.path.join(d, "t.cpp"), os.path.join(d, "t")
    open(src, "w").write(PROGRAM)
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, src, "-o", exe], check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout.splitlines()
    shutil.rmtree(d)
    return json.loads(out[0]), json.loads(out[1])


def test_diagonal_steps_cover_the_grid_in_dependency_order(output):
    cases, _ = output
    for c in cases:
        L, n = c["L"], c["n_seg"]
        assert len(c["steps"]) == L + n - 1
        seen = {}
        for i, (lo, hi, s_lo, *_rest) in enumerate(c["steps"]):
            assert 0 <= lo <= hi < L
            for l in range(lo, hi + 1):
                s = s_lo - (l - lo)
                assert 0 <= s < n and l + s == i
                assert (l, s) not in seen
                seen[(l, s)] = i
        assert len(seen) == L * n
        for (l, s), i in seen.items():
            if l > 0:
                assert seen[(l - 1, s)] < i
            if s > 0:
                assert seen[(l, s - 1)] < i
            if l + 1 < L and s + 1 < n:   # as many cells per step as the grid allows
                assert lo <= hi


def test_short_last_segment_and_its_cell(output):
    cases, _ = output
    for c in cases:
        S, n, n_tok = c["S"], c["n_seg"], c["n_tok"]
        assert (n - 1) * S < n_tok <= n * S and c["last_len"] == n_tok - (n - 1) * S
        for (lo, hi, s_lo, l_last, _r, _y) in c["steps"]:
            cells = {s_lo - (l - lo): l for l in range(lo, hi + 1)}
            if n - 1 in cells:
                assert l_last == cells[n - 1]
            else:
                assert not (lo <= l_last <= hi)


def test_results_final_after_each_step(output):
    cases, _ = output
    for c in cases:
        L, S, n, n_tok = c["L"], c["S"], c["n_seg"], c["n_tok"]
        done = set()
        prev_rows = prev_layers = 0
        for i, (lo, hi, s_lo, _l, rows, layers) in enumerate(c["steps"]):
            done |= {(l, s_lo - (l - lo)) for l in range(lo, hi + 1)}
            segs_out = [s for s in range(n) if (L - 1, s) in done]          # left the last layer
            layers_out = [l for l in range(L) if (l, n - 1) in done]        # ran their last segment
            assert segs_out == list(range(len(segs_out))) and layers_out == list(range(len(layers_out)))
            assert rows == min(n_tok, len(segs_out) * S) and layers == len(layers_out)
            assert rows >= prev_rows and layers >= prev_layers
            prev_rows, prev_layers = rows, layers
        assert prev_rows == n_tok and prev_layers == L
        seq = c["seq"]
        assert [r for r, _ in seq] == [min(n_tok, (s + 1) * S) for s in range(n)]
        assert [y for _, y in seq] == [0] * (n - 1) + [L]


def test_pair_tile_rule(output):
    _, pairs = output
    # 1040-row cells (one sequence, 1024 + 16 rows) and batches of 2 and 4 stay on single-CTA tiles;
    # row counts that fill 256-row tiles (LM head chunks, long sequences, batches of 8+) use pairs
    assert {int(k): v for k, v in pairs.items()} == {16: 0, 128: 0, 200: 1, 256: 1, 300: 0, 1040: 0,
                                                     2080: 0, 4160: 0, 8192: 1, 8320: 1, 16640: 1,
                                                     131072: 1}
