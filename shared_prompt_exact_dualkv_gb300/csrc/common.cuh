// Packed shared-prompt layout and the per-launch tile schedule.
//
// Packed rows (DualKV abstract: P + N*R tokens instead of N*(P+R)): a group
// is its prompt followed by its N responses; a launch may hold several
// groups (micro-batches of several prompts, research-map page "Key
// results": mb=8).  Work is cut into 128-row tiles that never straddle a
// segment; the host lists them longest-first (each response's items
// together) in the launch parameters.
#pragma once

#include <cstdint>

namespace dkv {

constexpr int kTile = 128;          // rows per q tile and per kv tile
constexpr int kMaxSeg = 1040;       // segments (prompts + responses) per launch
constexpr int kMaxItems = 4096;     // work items per launch; longer lists run in several launches

// A work item: tile index inside its segment, the segment, and, for the
// dK/dV kernel, the sequence-chunk split of a prompt key tile.
__host__ __device__ constexpr uint32_t make_item(uint32_t tile, uint32_t seg, uint32_t split) {
  return tile | (seg << 16) | (split << 27);
}
__host__ __device__ constexpr uint32_t item_tile(uint32_t it) { return it & 0xFFFFu; }
__host__ __device__ constexpr uint32_t item_seg(uint32_t it) { return (it >> 16) & 0x7FFu; }
__host__ __device__ constexpr uint32_t item_split(uint32_t it) { return it >> 27; }

// Packed rows are cut into segments: every prompt group is its prompt
// segment followed by its response segments, and groups follow one another.
// info[s]: bits 0..15 = the prompt segment of s's group (s itself for a
// prompt); bits 16..31 = the group's number of responses (prompt segments).
struct Sched {
  int32_t T, Hq, Hkv, group;        // group = Hq / Hkv
  int32_t num_items;
  int32_t num_splits;               // dK/dV kernel: sequence chunks per prompt key tile
  int32_t nseg;
  int32_t acc_rows;                 // prompt rows in all groups (fp32 accumulator rows)
  float scale;                      // softmax scale
  float scale_log2;                 // softmax scale * log2(e)
  int32_t heads_outer;              // query-tile kernels: block b is head b / num_items, item b % num_items
                                    // (0: item b / heads, head b % heads)
  int32_t pq_lo, pq_hi;             // prompt query tiles [pq_lo, pq_hi) of every prompt take part
                                    // (0, 0xFFFF = all; a rank of a sharded step takes a part)
  int32_t off[kMaxSeg + 1];         // segment s is packed rows [off[s], off[s+1])
  int32_t info[kMaxSeg];
  int32_t acc_row[kMaxSeg];         // prompt segments: first row in the prompt accumulators
  uint32_t items[kMaxItems];

  __host__ __device__ int32_t prompt_of(int32_t seg) const { return info[seg] & 0xFFFF; }
  __host__ __device__ int32_t responses_of(int32_t pseg) const { return info[pseg] >> 16; }
  __host__ __device__ int32_t seg_tiles(int32_t seg) const { return (off[seg + 1] - off[seg] + kTile - 1) / kTile; }
};

// Key-tile walk of one query tile (forward and dQ).  A prompt query tile
// qt sees its own prompt's key tiles 0..qt (the last one masked causally).
// A query tile of a response first walks its group's whole prompt (region A,
// no mask except keys past the prompt in a ragged last tile), then its own
// response's key tiles 0..qt (region B, the last one masked causally).
struct KeyWalk {
  int32_t nA;       // key tiles in region A
  int32_t n;        // total key tiles
  int32_t q0;       // first packed row of the query tile
  int32_t q_end;    // end of the query tile's segment (rows >= q_end are not stored)
  int32_t kA0;      // first packed row of the group's prompt
  int32_t plen;     // prompt length of the group
  int32_t kB0;      // first packed row of region B (own response start)

  __device__ __forceinline__ void init(const Sched& s, uint32_t item) {
    const int32_t tile = static_cast<int32_t>(item_tile(item));
    const int32_t seg = static_cast<int32_t>(item_seg(item));
    const int32_t ps = s.prompt_of(seg);
    kA0 = s.off[ps];
    plen = s.off[ps + 1] - kA0;
    q_end = s.off[seg + 1];
    if (ps == seg) {
      nA = 0;
      kB0 = kA0;
      n = tile + 1;
    } else {
      nA = (plen + kTile - 1) / kTile;
      kB0 = s.off[seg];
      n = nA + tile + 1;
    }
    q0 = kB0 + tile * kTile;
  }
  // First packed key row of key tile j.
  __device__ __forceinline__ int32_t k0(int32_t j) const {
    return j < nA ? kA0 + j * kTile : kB0 + (j - nA) * kTile;
  }
  // 0: no mask; 1: causal diagonal (col > row masked); 2: keys past the prompt masked.
  __device__ __forceinline__ int32_t mask_kind(int32_t j) const {
    if (j == n - 1) return 1;
    if (j == nA - 1 && (plen % kTile) != 0) return 2;
    return 0;
  }
  // For mask kind 2: columns >= this are past the prompt.
  __device__ __forceinline__ int32_t key_limit(int32_t j) const { return kA0 + plen - k0(j); }
};

}  // namespace dkv
