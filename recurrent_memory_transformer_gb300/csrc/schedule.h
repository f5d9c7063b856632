// Host-side arithmetic of the two cell schedules (plain C++, no CUDA).
//
// Summary page of "Diagonal Batching Unlocks Parallelism in Recurrent Memory
// Transformers for Long Contexts", section 二: cell (l, s) depends on
// (l-1, s) and (l, s-1), so every cell with l + s = i runs in grouped step i;
// L + n - 1 steps cover the L x n grid.  The cells of step i are the
// contiguous layer range [lo, hi] with segment s = i - l, i.e. segment
// s_lo = i - lo for layer lo and one segment less per layer above it.
// The sequential schedule runs one cell per step: segment by segment, layer
// by layer.  The library's forward loops, the launch count and the host-copy
// bookkeeping all use these functions; tests/test_schedule_cpu.py compiles
// this header alone and checks them against the grid's properties.
#pragma once

#include <stdint.h>

namespace armt {

struct CellRange {
  int lo, hi;     // layers of the step's cells
  int64_t s_lo;   // segment of the cell of layer lo; layer l runs segment s_lo - (l - lo)
};

// Step i (0 <= i < L + n - 1) of the diagonal schedule over L layers, n segments.
inline CellRange diagonal_step(int64_t i, int L, int64_t n) {
  CellRange r;
  r.lo = (int)(i - n + 1 > 0 ? i - n + 1 : 0);
  r.hi = (int)(i < L - 1 ? i : L - 1);
  r.s_lo = i - r.lo;
  return r;
}

inline int64_t diagonal_steps(int L, int64_t n) { return L + n - 1; }

// Segments and the last one's length for n_tok tokens in segments of S.
inline int64_t n_segments_for(int64_t n_tok, int S) { return (n_tok + S - 1) / S; }
inline int last_segment_len(int64_t n_tok, int S) {
  return (int)(n_tok - (n_segments_for(n_tok, S) - 1) * S);
}

// Layer of the cell that runs the last segment (n - 1) within a step whose
// layer lo runs segment s_lo; it belongs to the step when lo <= it <= hi.
inline int64_t last_segment_layer(int lo, int64_t s_lo, int64_t n) { return lo + (s_lo - (n - 1)); }

// After diagonal step i: hidden rows final (segments 0..i-L+1 have left the
// last layer; at most n_tok) and layers whose state is final (layers
// 0..i-n+1 have run their last segment).
inline int64_t diagonal_rows_final(int64_t i, int L, int S, int64_t n_tok) {
  const int64_t segs = i - L + 2 > 0 ? i - L + 2 : 0;
  return segs * S < n_tok ? segs * S : n_tok;
}
inline int diagonal_layers_final(int64_t i, int64_t n) { return (int)(i - n + 2 > 0 ? i - n + 2 : 0); }

// Sequential schedule, after segment s has run through all L layers.
inline int64_t sequential_rows_final(int64_t s, int S, int64_t n_tok) {
  return (s + 1) * S < n_tok ? (s + 1) * S : n_tok;
}
inline int sequential_layers_final(int64_t s, int64_t n, int L) { return s == n - 1 ? L : 0; }

// CTA-pair tiles cover 256 rows, single-CTA tiles 128: the pair kernel is
// chosen when it pads `rows` at most 3 % more than 128-row tiles do.
inline bool pair_tiles_pay_off(long long rows) {
  const long long p = (rows + 255) / 256 * 256, s1 = (rows + 127) / 128 * 128;
  return p * 100 <= s1 * 103;
}

}  // namespace armt
