// Packed shared-prompt layout and the per-launch tile schedule.
//
// Packed rows (DualKV abstract: P + N*R tokens instead of N*(P+R)): the
// prompt is rows [0, P); response i is rows [off[i], off[i+1]) with off[0] = P
// and off[N] = T.  Work is cut into 128-row tiles that never straddle a
// segment; the host lists them longest-first in the launch parameters.
#pragma once

#include <cstdint>

namespace dkv {

constexpr int kTile = 128;          // rows per q tile and per kv tile
constexpr int kMaxSeq = 1024;       // N limit (offsets live in the launch parameters)
constexpr int kMaxItems = 5600;     // work items per launch (parameter space bound)

// A work item: tile index inside its segment, the segment (0 = prompt,
// i + 1 = response i) and, for the dK/dV kernel, the sequence-chunk split.
__host__ __device__ constexpr uint32_t make_item(uint32_t tile, uint32_t seg, uint32_t split) {
  return tile | (seg << 16) | (split << 27);
}
__host__ __device__ constexpr uint32_t item_tile(uint32_t it) { return it & 0xFFFFu; }
__host__ __device__ constexpr uint32_t item_seg(uint32_t it) { return (it >> 16) & 0x7FFu; }
__host__ __device__ constexpr uint32_t item_split(uint32_t it) { return it >> 27; }

struct Sched {
  int32_t T, P, N, Hq, Hkv, group;  // group = Hq / Hkv
  int32_t num_items;
  int32_t num_splits;               // dK/dV kernel: sequence chunks per prompt kv tile
  float scale;                      // softmax scale
  float scale_log2;                 // softmax scale * log2(e)
  int32_t off[kMaxSeq + 1];
  uint32_t items[kMaxItems];
};

// Key-tile walk of one query tile (forward and dQ).  A prompt query tile
// qt sees prompt key tiles 0..qt (the last one masked causally).  A query
// tile of response i first walks the whole prompt (region A, no mask except
// keys >= P in a ragged last tile), then its own response's key tiles
// 0..qt (region B, the last one masked causally).
struct KeyWalk {
  int32_t nA;       // key tiles in region A
  int32_t n;        // total key tiles
  int32_t q0;       // first packed row of the query tile
  int32_t q_end;    // end of the query tile's segment (rows >= q_end are not stored)
  int32_t kB0;      // first packed row of region B (own response start)
  int32_t P;

  __device__ __forceinline__ void init(const Sched& s, uint32_t item) {
    const int32_t tile = static_cast<int32_t>(item_tile(item));
    const int32_t seg = static_cast<int32_t>(item_seg(item));
    P = s.P;
    if (seg == 0) {
      nA = 0;
      kB0 = 0;
      q0 = tile * kTile;
      q_end = s.P;
      n = tile + 1;
    } else {
      nA = (s.P + kTile - 1) / kTile;
      kB0 = s.off[seg - 1];
      q0 = kB0 + tile * kTile;
      q_end = s.off[seg];
      n = nA + tile + 1;
    }
  }
  // First packed key row of key tile j.
  __device__ __forceinline__ int32_t k0(int32_t j) const {
    return j < nA ? j * kTile : kB0 + (j - nA) * kTile;
  }
  // 0: no mask; 1: causal diagonal (col > row masked); 2: keys >= P masked.
  __device__ __forceinline__ int32_t mask_kind(int32_t j) const {
    if (j == n - 1) return 1;
    if (j == nA - 1 && (P % kTile) != 0) return 2;
    return 0;
  }
};

}  // namespace dkv
