// Launch plan of one product of the backward pass (host only): the tile and
// the split of K.  Kept apart from the kernels so that it can be checked on
// a machine without a GPU.
#pragma once

#include <algorithm>

namespace armt {

// How one product of the backward is launched: the tile (128 x 128 where
// that still gives every SM a block, else 64 x 64) and, for products with
// fewer tiles than SMs and K >= 128, a split of K into ksplit chunks of kchunk
// (a multiple of 16; about two blocks per SM; bounded by the partial-product
// scratch of part_cap floats).  ksplit = 1: no split.
struct BwGemmPlan {
  int bm = 64;
  int ksplit = 1, kchunk = 0;
};

inline BwGemmPlan bw_gemm_plan(int M, int N, int K, int groups, int num_sms, long long part_cap) {
  BwGemmPlan p;
  const long long tiles128 = (long long)((N + 127) / 128) * ((M + 127) / 128) * groups;
  p.bm = (M >= 128 && N >= 128 && tiles128 >= num_sms) ? 128 : 64;
  const long long tiles = (long long)((N + p.bm - 1) / p.bm) * ((M + p.bm - 1) / p.bm) * groups;
  int ks = 1;
  if (tiles < num_sms && K >= 128) {
    ks = (int)std::min<long long>((2LL * num_sms + tiles - 1) / tiles, K / 64);
    while (ks > 1 && (long long)ks * groups * M * N > part_cap) --ks;
  }
  if (ks > 1) {
    p.kchunk = ((K + ks - 1) / ks + 15) / 16 * 16;
    p.ksplit = (K + p.kchunk - 1) / p.kchunk;
  }
  return p;
}

// Adjoints handed between reverse diagonals live in two buffers used by
// parity.  Reverse diagonal i (cells (l, i - l)) reads the adjoint of its
// cells' output rows (written by cell (l + 1, s) on diagonal i + 1) and of the
// state each cell wrote (handed on by cell (l, s + 1) on diagonal i + 1) from
// buffer bw_in_buf(i), and writes its cells' input-row adjoints (slot l - 1)
// and entry-state adjoints (slot l) into bw_out_buf(i), which diagonal i - 1
// reads.  The final state's adjoints enter layer l's first cell in reverse
// order, (l, n - 1) on diagonal l + n - 1; the initial state's adjoints leave
// layer l's cell (l, 0) on diagonal l.
inline int bw_in_buf(long long i) { return (int)(i & 1); }
inline int bw_out_buf(long long i) { return (int)((i + 1) & 1); }
inline int bw_state_seed_buf(int l, long long n) { return bw_in_buf(l + n - 1); }
inline int bw_state_result_buf(int l) { return bw_out_buf(l); }

}  // namespace armt
