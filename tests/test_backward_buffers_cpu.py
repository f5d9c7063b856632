"""The backward's hand-over buffers between reverse diagonals (csrc/bw_plan.h).

Reverse diagonal i of the backward (cells (l, i - l), run together) reads
two kinds of adjoints written by the diagonal before it (i + 1): those of its
cells' output rows (from cell (l + 1, s)) and those of the state each cell
wrote (from cell (l, s + 1)), and writes its cells' input-row adjoints (for
cell (l - 1, s)) and entry-state adjoints (for cell (l, s - 1)).  Two buffers
by parity hold them.  This test compiles the parity rules alone and replays
every backward of a set of grids on the host, with each buffer slot holding
the name of the cell that wrote it:
  * every cell reads exactly the adjoints its producer wrote (the final
    state's adjoints for the last segment of each layer);
  * nothing is overwritten before it has been read, and no diagonal reads a
    buffer it also writes;
  * after diagonal 0 the initial state's adjoints of layer l are where they
    are collected from.
(The recurrence's dependencies, section 二 of the summary page of "Diagonal
Batching Unlocks Parallelism in Recurrent Memory Transformers for Long
Contexts": cell (l, s) needs (l - 1, s) and (l, s - 1); the adjoint runs them
in reverse.)
"""
import json
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "recurrent_memory_transformer_gb300", "csrc")

GRIDS = [(1, 1), (1, 5), (2, 1), (2, 4), (3, 5), (4, 12), (16, 3), (16, 8), (5, 2)]

PROGRAM = r"""
#include <cstdio>
#include "bw_plan.h"
int main() {
  int L; long long n;
  std::printf("[");
  bool first = true;
  while (std::scanf("%d %lld", &L, &n) == 2) {
    std::printf("%s{\"L\":%d,\"n\":%lld,\"in\":[", first ? "" : ",", L, n);
    first = false;
    for (long long i = 0; i < L + n - 1; ++i) std::printf("%s%d", i ? "," : "", armt::bw_in_buf(i));
    std::printf("],\"out\":[");
    for (long long i = 0; i < L + n - 1; ++i) std::printf("%s%d", i ? "," : "", armt::bw_out_buf(i));
    std::printf("],\"seed\":[");
    for (int l = 0; l < L; ++l) std::printf("%s%d", l ? "," : "", armt::bw_state_seed_buf(l, n));
    std::printf("],\"result\":[");
    for (int l = 0; l < L; ++l) std::printf("%s%d", l ? "," : "", armt::bw_state_result_buf(l));
    std::printf("]}");
  }
  std::printf("]\n");
  return 0;
}
"""


@pytest.fixture(scope="module")
def rules():
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    with tempfile.TemporaryDirectory() as td:
        src, exe = os.path.join(td, "bufs.cpp"), os.path.join(td, "bufs")
        open(src, "w").write(PROGRAM)
        r = subprocess.run([cxx, "-std=c++17", "-I", CSRC, "-o", exe, src], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
        inp = "\n".join(f"{L} {n}" for L, n in GRIDS)
        out = subprocess.run([exe], input=inp, capture_output=True, text=True, check=True).stdout
    return json.loads(out)


def test_every_cell_reads_what_its_producer_wrote(rules):
    for g in rules:
        L, n = g["L"], g["n"]
        rows = [{}, {}]    # buffer -> slot -> (writer, read yet)
        state = [{}, {}]
        for l in range(L):
            state[g["seed"][l]][l] = [("final", l), False]
        for i in reversed(range(L + n - 1)):
            cin, cout = g["in"][i], g["out"][i]
            assert cin != cout, (L, n, i)
            cells = [(l, i - l) for l in range(L) if 0 <= i - l < n]
            # every read of the diagonal, then every write (they use different buffers)
            for l, s in cells:
                if l < L - 1:
                    who, _ = rows[cin][l]
                    assert who == ("rows", l + 1, s), (L, n, l, s, who)
                    rows[cin][l][1] = True
                want = ("state", l, s + 1) if s < n - 1 else ("final", l)
                who, _ = state[cin][l]
                assert who == want, (L, n, l, s, who)
                state[cin][l][1] = True
            for l, s in cells:
                if l > 0:
                    prev = rows[cout].get(l - 1)
                    assert prev is None or prev[1], (L, n, l, s, prev)   # nothing unread is lost
                    rows[cout][l - 1] = [("rows", l, s), False]
                prev = state[cout].get(l)
                assert prev is None or prev[1], (L, n, l, s, prev)
                state[cout][l] = [("state", l, s), False]
        for l in range(L):
            who, _ = state[g["result"][l]][l]
            assert who == ("state", l, 0), (L, n, l, who)
