"""Host-side task list of the persistent wavefront (csrc/wavefront.cuh).

The persistent kernel takes tasks in list order and a task waits for the
(cell, stage) counters it depends on, so it can never deadlock as long as
every dependency is satisfied by tasks that come earlier in the list.  This
test compiles the task builder alone (host code, no GPU) and checks, for
several grids and a short last segment:
  * every dependency's counter is completed only by earlier tasks, and the
    count a task waits for equals the number of tasks of that counter;
  * a cell's first stage waits for the previous cell of its layer and the
    same segment's cell one layer down (section 二 of the summary page of
    "Diagonal Batching Unlocks Parallelism in Recurrent Memory Transformers
    for Long Contexts": cell (l, s) needs (l-1, s) and (l, s-1));
  * every stage that applies to a cell appears, once per block.
"""
import json
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "recurrent_memory_transformer_gb300", "csrc")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

PROGRAM = r"""
#include <cstdio>
#include "wavefront.cuh"
using namespace armt;
int main() {
  struct Case { int L; long long n; int last_len; };
  const Case cases[] = {{1, 1, 16}, {2, 4, 16}, {3, 5, 11}, {4, 12, 16}, {16, 3, 7}};
  std::printf("[");
  bool firstc = true;
  for (const Case& c : cases) {
    WfArgs a{};
    a.T = 20; a.S = 16; a.M = 4; a.d = 64; a.k = 16; a.Hq = 2; a.nw = 96; a.L = c.L;
    a.upd_rows = 32; a.n_seg = c.n; a.last_len = c.last_len;
    auto g = [](int N, int rows) { WfGemm r{}; r.N = N; r.rows = rows; r.nbx = (N + 63) / 64; return r; };
    a.gq = g(16, 20); a.gr = g(64, 20); a.gqkv = g(192, 20); a.go = g(64, 20); a.ggu = g(256, 20);
    a.gd = g(64, 20); a.gw = g(96, 4);
    std::vector<WfTask> t = wf_tasks(a, c.n);
    std::printf("%s{\"L\":%d,\"n\":%lld,\"last_len\":%d,\"nstage\":%d,\"tasks\":[", firstc ? "" : ",", c.L, c.n,
                c.last_len, (int)WF_NSTAGE);
    firstc = false;
    for (size_t i = 0; i < t.size(); ++i)
      std::printf("%s[%d,%d,%d,%d,%d,%d,%d,%d,%d,%d,%d]", i ? "," : "", t[i].stage, t[i].l, t[i].s, t[i].block,
                  t[i].self, t[i].dep[0], t[i].need[0], t[i].dep[1], t[i].need[1], t[i].dep[2], t[i].need[2]);
    std::printf("]}");
  }
  std::printf("]\n");
  return 0;
}
"""


@pytest.fixture(scope="module")
def cases():
    if not os.path.exists(NVCC) and shutil.which("nvcc") is None:
        pytest.skip("nvcc not available")
    nvcc = NVCC if os.path.exists(NVCC) else shutil.which("nvcc")
    with tempfile.TemporaryDirectory() as td:
        src = os.path.join(td, "wf.cu")
        exe = os.path.join(td, "wf")
        open(src, "w").write(PROGRAM)
        r = subprocess.run([nvcc, "-std=c++17", "-I", CSRC, "-o", exe, src], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout
    return json.loads(out)


def test_dependencies_point_to_earlier_tasks_with_exact_counts(cases):
    for c in cases:
        first_idx, last_idx, count = {}, {}, {}
        for i, t in enumerate(c["tasks"]):
            self_ = t[4]
            first_idx.setdefault(self_, i)
            last_idx[self_] = i
            count[self_] = count.get(self_, 0) + 1
        for i, t in enumerate(c["tasks"]):
            for dep, need in ((t[5], t[6]), (t[7], t[8]), (t[9], t[10])):
                if dep < 0:
                    continue
                assert dep in count, (c["L"], c["n"], i, dep)
                assert last_idx[dep] < i, (c["L"], c["n"], i, dep)     # all of it comes earlier
                assert need == count[dep], (c["L"], c["n"], i, dep, need, count[dep])


def test_first_stage_waits_for_both_grid_neighbours(cases):
    for c in cases:
        L, n, ns = c["L"], c["n"], c["nstage"]
        upd, depi = 18, 14  # WF_UPD, WF_DEPI
        for t in c["tasks"]:
            stage, l, s = t[0], t[1], t[2]
            first = (stage == 0) if l == 0 else (stage == 1)   # gather for layer 0, else the query product
            if not first:
                continue
            deps = {d for d in (t[5], t[7], t[9]) if d >= 0}
            if s > 0:
                assert (l * n + s - 1) * ns + upd in deps, (l, s)
            if l > 0:
                assert (((l - 1) * n + s) * ns + depi) in deps, (l, s)


def test_every_applicable_stage_appears_once_per_block(cases):
    for c in cases:
        L, n = c["L"], c["n"]
        seen = {}
        for t in c["tasks"]:
            seen.setdefault((t[1], t[2], t[0]), set()).add(t[3])
        for l in range(L):
            for s in range(n):
                stages = {st for (ll, ss, st) in seen if ll == l and ss == s}
                want = set(range(1, 19)) | ({0} if l == 0 else set()) | ({19} if l == L - 1 else set())
                assert stages == want, (l, s, sorted(stages))
                for st in stages:
                    blocks = seen[(l, s, st)]
                    assert blocks == set(range(len(blocks))), (l, s, st)
        # the final norm of a short last segment covers only its rows
        if c["last_len"] < 16:
            assert len(seen[(L - 1, n - 1, 19)]) == c["last_len"]
