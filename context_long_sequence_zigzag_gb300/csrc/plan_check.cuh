// plan_check.cuh — debug-mode consistency checks of a tile plan entry
// against the buffers a CTA will touch (every TMA coordinate, output row and
// loop bound of the attention kernels is derived from these fields).
//
// With debug checks on (cp_set_debug_checks), thread 0 of every attention
// CTA checks its plan entry before any TMA load, TMEM allocation or store;
// a bad entry records 0x200 | site in the device error word and the whole
// CTA returns without touching memory.  The host runs the same function over
// every plan it uploads.  Nothing traps: a failure is a status the host reads.
#pragma once

#include "internal.h"

namespace cpattn {

enum : int32_t {
  kErrPlanBase = 0x200,  // | site: which check of plan_entry_check failed
  kPlanTileIndex = 1,
  kPlanHead = 2,
  kPlanTileRows = 3,
  kPlanOutRows = 4,
  kPlanRangeList = 5,
  kPlanRangeRows = 6,
  kPlanWork = 7,
  kPlanPack = 8,
};

// A gathered key tile (run r): its pieces tile the rows [0, kTile) in order
// from 8-row boundaries, load rows that start inside the tensors, and its key
// mask is exactly the union of the pieces' key rows.
__host__ __device__ inline bool pack_entry_ok(const PackMask* packs, int32_t num_packs, const PackPiece* pieces,
                                              int32_t num_pieces, const RangeDesc& r, int64_t range_rows) {
  const int32_t count = r.flags >> kPackCountShift;
  if (packs == nullptr || pieces == nullptr || r.pos0 < 0 || r.pos0 >= num_packs) return false;
  if (count < 1 || count > kTile / 8 || r.row0 < 0 || int64_t(r.row0) + count > num_pieces) return false;
  const PackMask pk = packs[r.pos0];
  uint32_t want[4] = {0u, 0u, 0u, 0u};
  int32_t next = 0;
  for (int i = 0; i < count; ++i) {
    const PackPiece pc = pieces[r.row0 + i];
    if (pc.dst != next || pc.rows < 8 || (pc.rows & 7) || pc.dst + pc.rows > kTile) return false;
    if (pc.keys < 1 || pc.keys > pc.rows || pc.src < 0 || int64_t(pc.src) + pc.keys > range_rows) return false;
    for (int w = 0; w < 4; ++w) {  // rows [dst, dst + keys) of word w, without indexing by a variable
      const int lo = pc.dst > 32 * w ? pc.dst : 32 * w;
      const int hi = pc.dst + pc.keys < 32 * w + 32 ? pc.dst + pc.keys : 32 * w + 32;
      if (hi > lo) want[w] |= (hi - lo == 32 ? 0xffffffffu : (1u << (hi - lo)) - 1u) << (lo - 32 * w);
    }
    next = pc.dst + pc.rows;
  }
  if (next != kTile) return false;
  for (int w = 0; w < 4; ++w)
    if (pk.valid[w] != want[w]) return false;
  return true;
}

// 0 when the entry is consistent, else the number of the failed check.
//   tile_rows  : rows of the tensors the tile indexes (q for query-major
//                plans, k / v for key-major ones)
//   range_rows : rows of the tensors the runs index
//   packs, pieces : the gathered key tiles (null / 0 for plans without them)
__host__ __device__ inline int plan_entry_check(const TileDesc* tiles, int32_t num_tiles, const RangeDesc* ranges,
                                                int32_t num_ranges, const PackMask* packs, int32_t num_packs,
                                                const PackPiece* pieces, int32_t num_pieces, int tile_idx, int head,
                                                int heads, int kv_head, int kv_heads, int64_t tile_rows,
                                                int64_t range_rows, int32_t block_mode, int64_t out_rows) {
  if (tile_idx < 0 || tile_idx >= num_tiles) return kPlanTileIndex;
  if (head < 0 || head >= heads || kv_head < 0 || kv_head >= kv_heads) return kPlanHead;
  const TileDesc t = tiles[tile_idx];
  if (t.nrows < 1 || t.nrows > kTile || t.row0 < 0 || int64_t(t.row0) + t.nrows > tile_rows) return kPlanTileRows;
  if (block_mode && (t.out_row0 < 0 || int64_t(t.out_row0) + t.nrows > out_rows)) return kPlanOutRows;
  if (t.range_begin < 0 || t.range_count < 0 || int64_t(t.range_begin) + t.range_count > num_ranges)
    return kPlanRangeList;
  int64_t steps = 0;
  for (int i = 0; i < t.range_count; ++i) {
    const RangeDesc r = ranges[t.range_begin + i];
    if (r.flags & kRangePacked) {
      if (r.nrows != kTile || (r.flags & kRangeMasked) ||
          !pack_entry_ok(packs, num_packs, pieces, num_pieces, r, range_rows))
        return kPlanPack;
    } else if (r.nrows < 1 || r.row0 < 0 || int64_t(r.row0) + r.nrows > range_rows) {
      return kPlanRangeRows;
    }
    steps += (r.nrows + kTile - 1) / kTile;
  }
  if (steps != t.work) return kPlanWork;
  return 0;
}

#ifdef __CUDACC__
// The CTA-wide form: thread 0 checks, every thread gets the verdict.  Returns
// false (after recording the error) when the CTA must not run.  Must be
// called by all threads of the CTA, before any barrier initialisation.
__device__ inline bool debug_plan_ok(const AttnArgs& a, int tile_idx, int head, int kv_head, bool key_major,
                                     int32_t* err) {
  int bad = 0;
  if (threadIdx.x == 0) {
    const int64_t tq = a.T, tkv = a.T_kv ? a.T_kv : a.T;
    bad = plan_entry_check(a.tiles, a.num_tiles, a.ranges, a.num_ranges, a.packs, a.num_packs, a.pieces,
                           a.num_pieces, tile_idx, head, key_major ? a.hkv : a.hq,
                           kv_head, a.hkv, key_major ? tkv : tq, key_major ? tq : tkv, a.block_mode, a.lse_stride);
    if (bad && err) atomicCAS(err, 0, kErrPlanBase | bad);
  }
  return __syncthreads_or(bad) == 0;
}
#endif

}  // namespace cpattn
