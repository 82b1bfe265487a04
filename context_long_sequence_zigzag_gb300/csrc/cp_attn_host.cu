// cp_attn_host.cu — host runtime of libcpattn: descriptor validation, the
// shard map, the per-call tile plans (ring visiting order, causal skipping),
// workspace layout and dispatch to the kernels.  Every exported function of
// include/cp_attn.h is defined here.
//
// The shard map and block classes follow
//   "Ulysses与Ring-Attention详解" §4.2 (zigzag: rank r holds chunk r and chunk
//   2C-1-r) and "超长上下文训练速度翻倍秘籍" §2 pitfall 1 / §3 varlen CP (own
//   diagonal block causal, earlier blocks unmasked, every packed sub-sequence
//   cut into CP pieces), and "LLM context parallel production guide",
//   "因果 Attention 会制造 Rank 负载不均" (blocks above the diagonal skipped).
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <list>
#include <map>
#include <memory>
#include <mutex>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "internal.h"
#include "plan_check.cuh"

namespace cpattn {
namespace {

// A named NVTX range around every entry point that enqueues GPU work, so that
// a profiler's timeline attributes kernels to calls (a no-op without one).
// The allocation-free forward has none: a profiler's NVTX handler may
// allocate.
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};

// One rank's run of one sequence, stored contiguously in sharded order.  Its
// tokens sit at global rows grow0, grow0 + stride, ... (stride 1 except for
// the striped layout, where it is C).
struct Chunk {
  int32_t seq, idx, pos0, len, rank;
  int64_t grow0;   // first global row
  int64_t srow0;   // first sharded row
  int32_t stride;  // global-row step between consecutive tokens of the chunk
};

struct ShardMap {
  int32_t C = 0, S = 0, per = 0;  // ranks, sequences, chunks per rank per sequence
  bool striped = false;
  std::vector<Chunk> chunks;      // index (r * S + s) * per + k
  std::vector<int64_t> rank_off;  // C + 1

  const Chunk& at(int r, int s, int k) const { return chunks[(size_t(r) * S + s) * per + k]; }
};

// Position of chunk X's first token in the coordinates of a (query chunk A,
// key chunk B) block.  Contiguous and zigzag chunks hold consecutive
// positions, so that is X.pos0.  A striped chunk of rank r holds positions
// r, r + C, r + 2C, ...: key j of rank rk is visible to query i of rank rq
// iff rk + C*j <= rq + C*i, i.e. iff j + [rk > rq] <= i.  Queries therefore
// take their index inside the chunk as position and keys of a higher rank
// are shifted by one; positions stay consecutive inside every chunk.
int32_t key_pos0(const ShardMap& m, const Chunk& key, const Chunk& query) {
  return m.striped ? (key.rank > query.rank ? 1 : 0) : key.pos0;
}
int32_t query_pos0(const ShardMap& m, const Chunk& query, const Chunk& key) {
  return m.striped ? (key.rank > query.rank ? -1 : 0) : query.pos0;
}

std::vector<int32_t> seqlens_of(const cp_desc_t* d) {
  std::vector<int32_t> cu;
  if (d->cu_seqlens == nullptr) {
    cu = {0, int32_t(d->total_tokens)};
  } else {
    cu.assign(d->cu_seqlens, d->cu_seqlens + d->num_seqs + 1);
  }
  return cu;
}

// Checks shared by every call that reads the shard map.
cp_status_t check_map_fields(const cp_desc_t* d) {
  if (d == nullptr) return CP_ERR_INVALID_ARG;
  if (d->total_tokens < 0 || d->total_tokens > INT32_MAX) return CP_ERR_INVALID_ARG;
  if (d->num_seqs < 1) return CP_ERR_INVALID_ARG;
  if (d->cp_size < 1 || d->cp_size > 4096) return CP_ERR_INVALID_ARG;
  if (d->layout != CP_LAYOUT_CONTIGUOUS && d->layout != CP_LAYOUT_ZIGZAG && d->layout != CP_LAYOUT_STRIPED)
    return CP_ERR_INVALID_ARG;
  if (d->cu_seqlens == nullptr) {
    if (d->num_seqs != 1) return CP_ERR_INVALID_ARG;
    return CP_OK;
  }
  const int32_t* cu = d->cu_seqlens;
  if (cu[0] != 0) return CP_ERR_INVALID_ARG;
  for (int s = 0; s < d->num_seqs; ++s)
    if (cu[s + 1] < cu[s]) return CP_ERR_INVALID_ARG;
  if (int64_t(cu[d->num_seqs]) != d->total_tokens) return CP_ERR_INVALID_ARG;
  return CP_OK;
}

cp_status_t check_attn_fields(const cp_desc_t* d) {
  cp_status_t st = check_map_fields(d);
  if (st != CP_OK) return st;
  if (d->hq < 1 || d->hkv < 1 || d->hq % d->hkv != 0) return CP_ERR_INVALID_ARG;
  if (d->d_qk < 1 || d->d_v < 1) return CP_ERR_INVALID_ARG;
  if (d->dtype != CP_DT_F32 && d->dtype != CP_DT_BF16) return CP_ERR_INVALID_ARG;
  if (d->gqa != CP_GQA_BLOCKED && d->gqa != CP_GQA_INTERLEAVED) return CP_ERR_INVALID_ARG;
  if (d->causal != 0 && d->causal != 1) return CP_ERR_INVALID_ARG;
  if (!(d->scale > 0.f) || !std::isfinite(d->scale)) return CP_ERR_INVALID_ARG;
  const int elt = d->dtype == CP_DT_BF16 ? 2 : 4;
  if ((d->d_qk * elt) % 16 != 0 || (d->d_v * elt) % 16 != 0) return CP_ERR_INVALID_ARG;
  // The CUDA-core path keeps head rows in registers spread over a warp.
  if (d->d_qk > 256 || d->d_v > 256) return CP_ERR_UNSUPPORTED;
  if (int64_t(d->total_tokens) * d->hq * std::max(d->d_qk, d->d_v) > (int64_t(1) << 40))
    return CP_ERR_UNSUPPORTED;
  return CP_OK;
}

ShardMap build_map(const cp_desc_t* d) {
  ShardMap m;
  std::vector<int32_t> cu = seqlens_of(d);
  m.C = d->cp_size;
  m.S = int32_t(cu.size()) - 1;
  m.per = d->layout == CP_LAYOUT_ZIGZAG ? 2 : 1;
  m.striped = d->layout == CP_LAYOUT_STRIPED;
  const int64_t n = int64_t(m.C) * m.per;  // pieces per sequence
  m.chunks.reserve(size_t(m.C) * m.S * m.per);
  m.rank_off.assign(m.C + 1, 0);
  int64_t srow = 0;
  for (int r = 0; r < m.C; ++r) {
    m.rank_off[r] = srow;
    for (int s = 0; s < m.S; ++s) {
      const int64_t L = int64_t(cu[s + 1]) - cu[s];
      if (m.striped) {
        Chunk ch;
        ch.seq = s;
        ch.idx = r;
        ch.pos0 = 0;  // block-relative positions: see key_pos0 / query_pos0
        ch.len = int32_t(L > r ? (L - r + m.C - 1) / m.C : 0);
        ch.rank = r;
        ch.grow0 = cu[s] + r;
        ch.srow0 = srow;
        ch.stride = m.C;
        m.chunks.push_back(ch);
        srow += ch.len;
        continue;
      }
      for (int k = 0; k < m.per; ++k) {
        const int64_t c = (k == 0) ? r : (2 * int64_t(m.C) - 1 - r);
        const int64_t lo = (c * L) / n, hi = ((c + 1) * L) / n;
        Chunk ch;
        ch.seq = s;
        ch.idx = int32_t(c);
        ch.pos0 = int32_t(lo);
        ch.len = int32_t(hi - lo);
        ch.rank = r;
        ch.grow0 = cu[s] + lo;
        ch.srow0 = srow;
        ch.stride = 1;
        m.chunks.push_back(ch);
        srow += hi - lo;
      }
    }
  }
  m.rank_off[m.C] = srow;
  return m;
}

// Position given to a merged run (two whole, unmasked zigzag chunks of one
// rank): keys far in the past (-kMergedPos) or queries far in the future
// (+kMergedPos), so that the kernels' causal tests see every pair visible.
constexpr int32_t kMergedPos = 1 << 29;

// Runs are merged only where positions stay far from kMergedPos.
bool merge_ok(const ShardMap& m, int seq) {
  if (m.per != 2) return false;
  int64_t len = 0;
  for (int r = 0; r < m.C; ++r) len += m.at(r, seq, 0).len + m.at(r, seq, 1).len;
  return len < kMergedPos / 4;
}

struct Plan {
  std::vector<TileDesc> tiles;
  std::vector<RangeDesc> ranges;
  std::vector<PackMask> packs;  // key masks of the gathered key tiles (kRangePacked runs)
  std::vector<PackPiece> pieces;
  std::vector<int32_t> tile_seq;  // key-major plans: each tile's sequence (host only, for the order)
  int32_t max_ranges = 0;
};

int32_t round8(int32_t n) { return (n + 7) & ~7; }

// Gathers the ragged tails of one tile's unmasked runs (key runs of a query
// tile, or query runs of a key tile) into shared tiles.  In an unmasked run
// every pair with the tile's rows is visible, so where a run's row sits in
// the tile it is cut into does not matter: each run keeps its whole
// kTile-row steps as a run of its own, and the tails (fewer than kTile rows
// each) are laid back to back from 8-row boundaries, split across two tiles
// where one fills up.  The rows between a tail's last row and the next
// boundary, and after the last tail up to the tile's end, are loaded from the
// rows that follow it and masked.  Done only where it saves tiles: where the
// tails would need as many tiles gathered as apart, nothing changes.  The
// tile's runs [first, end) of p.ranges become its masked and whole-step runs,
// in their order, followed by the gathered tiles.
void pack_tails(Plan& p, size_t first) {
  std::vector<RangeDesc> keep;
  std::vector<std::pair<int32_t, int32_t>> tails;  // (first sharded row, rows)
  for (size_t i = first; i < p.ranges.size(); ++i) {
    const RangeDesc r = p.ranges[i];
    if (r.flags != 0 || r.nrows % kTile == 0) {
      keep.push_back(r);
      continue;
    }
    const int32_t whole = r.nrows - r.nrows % kTile;
    if (whole > 0) keep.push_back(RangeDesc{r.row0, whole, r.pos0, 0});
    tails.emplace_back(r.row0 + whole, r.nrows - whole);
  }
  int32_t rows = 0;
  for (const auto& tl : tails) rows += round8(tl.second);
  if ((rows + kTile - 1) / kTile >= int32_t(tails.size())) return;  // no key tile saved
  p.ranges.resize(first);
  p.ranges.insert(p.ranges.end(), keep.begin(), keep.end());
  PackMask pk{};
  int32_t dst = 0, piece0 = 0, count = 0;
  auto close = [&]() {
    PackPiece& last = p.pieces.back();
    last.rows = kTile - last.dst;  // fill the tile with the rows that follow
    p.ranges.push_back(RangeDesc{piece0, kTile, int32_t(p.packs.size()), kRangePacked | (count << kPackCountShift)});
    p.packs.push_back(pk);
    dst = 0;
  };
  for (auto [src, n] : tails) {
    while (n > 0) {
      if (dst == 0) {
        pk = PackMask{};
        piece0 = int32_t(p.pieces.size());
        count = 0;
      }
      const int32_t take = std::min(n, kTile - dst);
      p.pieces.push_back(PackPiece{src, dst, round8(take), take});
      for (int32_t j = dst; j < dst + take; ++j) pk.valid[j >> 5] |= 1u << (j & 31);
      ++count;
      dst += round8(take);
      src += take;
      n -= take;
      if (dst == kTile) close();
    }
  }
  if (dst > 0) close();
}

int32_t ceil_tiles(int64_t n) { return int32_t((n + kTile - 1) / kTile); }

// Query-major plan: every query tile with the key runs it must visit, in ring
// order r, r-1, ..., r-C+1 (mod C).  q_rank / kv_rank >= 0 restrict the plan
// to one (query shard, key shard) block.  ring_step >= 0 gives one step of
// the transported ring instead: every rank's query tiles against the shard
// it holds at that step, rho = (r - step) mod C; from step 1 on that shard
// sits in the holder's slot of a ring buffer whose rank slots are slot_rows
// rows apart, and tiles that see nothing of it are left out.
Plan build_fwd_plan(const cp_desc_t* d, const ShardMap& m, int q_rank, int kv_rank, int ring_step = -1,
                    int64_t slot_rows = 0, bool pack = false) {
  Plan p;
  const bool causal = d->causal != 0;
  for (const Chunk& A : m.chunks) {
    if (q_rank >= 0 && A.rank != q_rank) continue;
    for (int32_t t0 = 0; t0 < A.len; t0 += kTile) {
      TileDesc t{};
      t.row0 = int32_t(A.srow0 + t0);
      t.nrows = std::min(kTile, A.len - t0);
      t.pos0 = A.pos0 + t0;
      t.rank = A.rank;
      t.out_row0 = q_rank >= 0 ? int32_t(t.row0 - m.rank_off[q_rank]) : t.row0;
      t.range_begin = int32_t(p.ranges.size());
      const int32_t qmin = t.pos0, qmax = t.pos0 + t.nrows - 1;
      int32_t work = 0;
      for (int step = 0; step < m.C; ++step) {
        const int rho = ((A.rank - step) % m.C + m.C) % m.C;
        if (kv_rank >= 0 && rho != kv_rank) continue;
        if (ring_step >= 0 && step != ring_step) continue;
        const size_t first = p.ranges.size();
        bool whole[2] = {false, false};  // run k covers its whole chunk without a mask
        for (int k = 0; k < m.per; ++k) {
          const Chunk& B = m.at(rho, A.seq, k);
          if (B.len == 0) continue;
          RangeDesc r{};
          const int32_t bpos = key_pos0(m, B, A);
          r.row0 = ring_step > 0 ? int32_t(A.rank * slot_rows + (B.srow0 - m.rank_off[rho])) : int32_t(B.srow0);
          r.pos0 = bpos;
          if (causal) {
            if (bpos > qmax) continue;  // entirely in the future: skipped
            r.nrows = std::min(B.len, qmax - bpos + 1);
            r.flags = (bpos + r.nrows - 1 > qmin) ? kRangeMasked : 0;
          } else {
            r.nrows = B.len;
            r.flags = 0;
          }
          whole[p.ranges.size() - first] = r.flags == 0 && r.nrows == B.len;
          p.ranges.push_back(r);
        }
        // A rank's two zigzag chunks of a sequence are adjacent rows: when the
        // tile sees both whole and unmasked they are one run (short chunks
        // then share key tiles).  Its keys are all visible, so it carries a
        // position far in the past instead of either chunk's.
        if (p.ranges.size() - first == 2 && whole[0] && whole[1] && merge_ok(m, A.seq) &&
            p.ranges[first + 1].row0 == p.ranges[first].row0 + p.ranges[first].nrows) {
          p.ranges[first].nrows += p.ranges[first + 1].nrows;
          p.ranges[first].pos0 = -kMergedPos;
          p.ranges.pop_back();
        }
        for (size_t i = first; i < p.ranges.size(); ++i) work += ceil_tiles(p.ranges[i].nrows);
      }
      if (pack) {
        pack_tails(p, size_t(t.range_begin));
        work = 0;
        for (size_t i = size_t(t.range_begin); i < p.ranges.size(); ++i) work += ceil_tiles(p.ranges[i].nrows);
      }
      t.range_count = int32_t(p.ranges.size()) - t.range_begin;
      t.work = work;
      if (ring_step > 0 && t.range_count == 0) continue;  // merging nothing would leave the accumulator as is
      p.max_ranges = std::max(p.max_ranges, t.range_count);
      p.tiles.push_back(t);
    }
  }
  return p;
}

// Key-major plan for the backward: every key tile with the query runs that
// see it, visiting ranks r, r+1, ... (the direction dK/dV travel in a ring).
Plan build_bwd_plan(const cp_desc_t* d, const ShardMap& m, bool pack = false) {
  Plan p;
  const bool causal = d->causal != 0;
  for (const Chunk& B : m.chunks) {
    for (int32_t t0 = 0; t0 < B.len; t0 += kTile) {
      TileDesc t{};
      t.row0 = int32_t(B.srow0 + t0);
      t.nrows = std::min(kTile, B.len - t0);
      t.pos0 = B.pos0 + t0;
      t.rank = B.rank;
      t.out_row0 = t.row0;
      t.range_begin = int32_t(p.ranges.size());
      const int32_t kmin = t.pos0, kmax = t.pos0 + t.nrows - 1;
      int32_t work = 0;
      for (int step = 0; step < m.C; ++step) {
        const int rho = (B.rank + step) % m.C;
        const size_t first = p.ranges.size();
        bool whole[2] = {false, false};  // run k covers its whole chunk without a mask
        for (int k = 0; k < m.per; ++k) {
          const Chunk& A = m.at(rho, B.seq, k);
          if (A.len == 0) continue;
          RangeDesc r{};
          const int32_t apos = query_pos0(m, A, B);
          if (causal) {
            if (apos + A.len - 1 < kmin) continue;  // every query precedes the keys
            const int32_t skip = std::max(0, kmin - apos);
            r.row0 = int32_t(A.srow0 + skip);
            r.nrows = A.len - skip;
            r.pos0 = apos + skip;
            r.flags = (r.pos0 < kmax) ? kRangeMasked : 0;
          } else {
            r.row0 = int32_t(A.srow0);
            r.nrows = A.len;
            r.pos0 = apos;
            r.flags = 0;
          }
          whole[p.ranges.size() - first] = r.flags == 0 && r.nrows == A.len;
          p.ranges.push_back(r);
        }
        // the two adjacent zigzag chunks of a rank as one query run when both
        // see the whole key tile (a position far in the future)
        if (p.ranges.size() - first == 2 && whole[0] && whole[1] && merge_ok(m, B.seq) &&
            p.ranges[first + 1].row0 == p.ranges[first].row0 + p.ranges[first].nrows) {
          p.ranges[first].nrows += p.ranges[first + 1].nrows;
          p.ranges[first].pos0 = kMergedPos;
          p.ranges.pop_back();
        }
        for (size_t i = first; i < p.ranges.size(); ++i) work += ceil_tiles(p.ranges[i].nrows);
      }
      if (pack) {  // the tails of the query runs that see the whole key tile
        pack_tails(p, size_t(t.range_begin));
        work = 0;
        for (size_t i = size_t(t.range_begin); i < p.ranges.size(); ++i) work += ceil_tiles(p.ranges[i].nrows);
      }
      t.range_count = int32_t(p.ranges.size()) - t.range_begin;
      t.work = work;
      p.max_ranges = std::max(p.max_ranges, t.range_count);
      p.tiles.push_back(t);
      p.tile_seq.push_back(B.seq);
    }
  }
  return p;
}

// Heaviest tiles first, so that the block scheduler starts the long ones
// early (longest-processing-time order).  A key-major plan of several
// sequences goes sequence by sequence instead (heaviest sequence first,
// heaviest tiles first inside each): its CTAs read the Q and dO of their
// own sequence, so the resident CTAs then share the Q and dO of a few
// sequences in L2 instead of touching every sequence's (in work order the
// dK/dV kernel read 5.7x its algorithmic bytes on a 128K-token pack of 16
// sequences).  With one sequence both orders are the same.
void order_by_work(Plan& p) {
  if (p.tile_seq.size() != p.tiles.size() || p.tiles.empty()) {
    std::stable_sort(p.tiles.begin(), p.tiles.end(),
                     [](const TileDesc& a, const TileDesc& b) { return a.work > b.work; });
    return;
  }
  const int32_t nseq = *std::max_element(p.tile_seq.begin(), p.tile_seq.end()) + 1;
  std::vector<int64_t> seq_work(size_t(nseq), 0);
  for (size_t i = 0; i < p.tiles.size(); ++i) seq_work[size_t(p.tile_seq[i])] += p.tiles[i].work;
  std::vector<size_t> idx(p.tiles.size());
  for (size_t i = 0; i < idx.size(); ++i) idx[i] = i;
  std::stable_sort(idx.begin(), idx.end(), [&](size_t a, size_t b) {
    const int32_t sa = p.tile_seq[a], sb = p.tile_seq[b];
    if (sa != sb) return seq_work[size_t(sa)] != seq_work[size_t(sb)] ? seq_work[size_t(sa)] > seq_work[size_t(sb)]
                                                                      : sa < sb;
    return p.tiles[a].work > p.tiles[b].work;
  });
  std::vector<TileDesc> tiles(p.tiles.size());
  std::vector<int32_t> seqs(p.tiles.size());
  for (size_t i = 0; i < idx.size(); ++i) {
    tiles[i] = p.tiles[idx[i]];
    seqs[i] = p.tile_seq[idx[i]];
  }
  p.tiles.swap(tiles);
  p.tile_seq.swap(seqs);
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t plan_bytes(const Plan& p) {
  return align256(p.tiles.size() * sizeof(TileDesc)) + align256(p.ranges.size() * sizeof(RangeDesc)) +
         align256(p.packs.size() * sizeof(PackMask)) + align256(p.pieces.size() * sizeof(PackPiece));
}

// Recently built plans.  A plan depends only on the shard map (T, the
// sequence lengths, C, the layout), the mask and which plan it is, so
// repeated calls on the same problem (every training step) reuse it instead
// of rebuilding it on the host; the upload into the call's workspace still
// happens every call, since the caller may use that memory for anything in
// between.
// kPlanQueryMajorPacked: the query-major plan with the unmasked runs' tails
// gathered into shared key tiles (the tensor-core forward and dQ kernels
// read those); kPlanKeyMajorPacked: the key-major plan with the tails of
// the query runs that see a whole key tile gathered into shared query tiles
// (the tensor-core dK/dV kernel with 128-row query steps).
enum PlanKind : int64_t { kPlanQueryMajor = 0, kPlanKeyMajor = 1, kPlanQueryMajorPacked = 2, kPlanKeyMajorPacked = 3 };
std::shared_ptr<const Plan> get_plan(const cp_desc_t* d, const ShardMap& m, PlanKind kind, int q_rank = -1,
                                     int kv_rank = -1, int ring_step = -1, int64_t slot_rows = 0) {
  static std::mutex mu;
  static std::list<std::pair<std::vector<int64_t>, std::shared_ptr<const Plan>>> cache;  // most recent first
  static size_t cached_bytes = 0;
  // a ring of C steps uses C plans; bounded by count and by host bytes
  constexpr size_t kMaxPlans = 80, kMaxBytes = size_t(256) << 20;
  std::vector<int64_t> key = {kind, q_rank, kv_rank, ring_step, slot_rows, d->total_tokens, d->cp_size, d->layout,
                              d->causal, d->num_seqs};
  if (d->cu_seqlens) key.insert(key.end(), d->cu_seqlens, d->cu_seqlens + d->num_seqs + 1);
  {
    std::lock_guard<std::mutex> lock(mu);
    for (auto it = cache.begin(); it != cache.end(); ++it)
      if (it->first == key) {
        cache.splice(cache.begin(), cache, it);
        return it->second;
      }
  }
  const bool key_major = kind == kPlanKeyMajor || kind == kPlanKeyMajorPacked;
  auto plan = std::make_shared<Plan>(key_major ? build_bwd_plan(d, m, kind == kPlanKeyMajorPacked)
                                               : build_fwd_plan(d, m, q_rank, kv_rank, ring_step, slot_rows,
                                                                kind == kPlanQueryMajorPacked));
  order_by_work(*plan);
  std::lock_guard<std::mutex> lock(mu);
  cache.emplace_front(std::move(key), plan);
  cached_bytes += plan_bytes(*plan);
  while (cache.size() > 1 && (cache.size() > kMaxPlans || cached_bytes > kMaxBytes)) {
    cached_bytes -= plan_bytes(*cache.back().second);
    cache.pop_back();
  }
  return plan;
}


// Host -> device copies of plans and tables go through a pinned staging
// ring, one per device.  From pageable memory the runtime may wait for the
// stream to drain before it stages a large copy (measured: a 128K-token varlen
// forward's ~0.7 MB plan held the calling thread for a whole earlier forward,
// 5.4 ms); from pinned memory the copy is queued and the call returns.  A
// region of the ring is reused only after the event recorded behind its last
// copy has completed.
class StagingRing {
 public:
  static constexpr size_t kBytes = size_t(32) << 20;
  static constexpr size_t kTracked = 64;

  // Queues dst <- src (bytes) on st through the ring of the current device;
  // false when the ring is not usable for this copy (the caller then copies
  // from the source directly).
  bool copy(void* dst, const void* src, size_t bytes, cudaStream_t st, cudaError_t* err) {
    if (bytes == 0 || bytes > kBytes / 4) return false;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(mu_);
    PerDevice& r = rings_[dev];
    if (r.failed) return false;
    if (!r.host) {
      if (cudaMallocHost(&r.host, kBytes) != cudaSuccess) {
        cudaGetLastError();
        r.host = nullptr;
        r.failed = true;
        return false;
      }
    }
    // at most kTracked copies tracked: the oldest has long finished by then
    while (r.inflight.size() >= kTracked) {
      cudaEventSynchronize(r.inflight.front().ev);
      r.free_events.push_back(r.inflight.front().ev);
      r.inflight.pop_front();
    }
    size_t off = align256(r.head);
    if (off + bytes > kBytes) off = 0;
    // wait for (normally long finished) copies still reading [off, off + bytes)
    for (auto it = r.inflight.begin(); it != r.inflight.end();) {
      if (it->begin < off + bytes && off < it->end) {
        cudaEventSynchronize(it->ev);
        r.free_events.push_back(it->ev);
        it = r.inflight.erase(it);
      } else {
        ++it;
      }
    }
    std::memcpy(static_cast<char*>(r.host) + off, src, bytes);
    *err = cudaMemcpyAsync(dst, static_cast<char*>(r.host) + off, bytes, cudaMemcpyHostToDevice, st);
    r.head = off + bytes;
    cudaEvent_t ev = nullptr;
    if (!r.free_events.empty()) {
      ev = r.free_events.back();
      r.free_events.pop_back();
    } else if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      ev = nullptr;
    }
    bool tracked = false;
    if (*err == cudaSuccess && ev) {
      if (cudaEventRecord(ev, st) == cudaSuccess) {
        r.inflight.push_back({off, off + bytes, ev});
        tracked = true;
      } else {
        cudaGetLastError();  // this failed record's own error (e.g. a stream of another device)
      }
    }
    if (!tracked) {
      // no completion to track: wait for the copy here before the region can
      // be reused (a failed copy leaves its error for the caller to read)
      if (*err == cudaSuccess) *err = cudaStreamSynchronize(st);
      if (ev) r.free_events.push_back(ev);
    }
    return true;
  }

 private:
  struct Span {
    size_t begin, end;
    cudaEvent_t ev;
  };
  struct PerDevice {
    void* host = nullptr;
    bool failed = false;
    size_t head = 0;
    std::list<Span> inflight;
    std::vector<cudaEvent_t> free_events;
  };
  std::mutex mu_;
  std::map<int, PerDevice> rings_;
};

// Held until the process exits (no destructor runs at exit, when the CUDA
// runtime may already be gone).
StagingRing& staging_ring() {
  static StagingRing* ring = new StagingRing();
  return *ring;
}

// dst <- src on st: through the staging ring when `pinned` allows it (every
// entry point but the allocation-free one), else straight from `src`, which
// must then stay valid until the runtime has staged it (it has when this
// returns).
cudaError_t h2d_async(void* dst, const void* src, size_t bytes, cudaStream_t st, bool pinned = true) {
  if (bytes == 0) return cudaSuccess;
  cudaError_t e = cudaSuccess;
  if (pinned && staging_ring().copy(dst, src, bytes, st, &e)) return e;
  return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, st);
}

// Copies the plan into the workspace at `base` (tiles, runs, gathered key
// tiles, their pieces, each from a 256-byte boundary) and points the kernel
// arguments at it.
cudaError_t upload_plan(const Plan& p, char* base, cudaStream_t st, AttnArgs& a, bool pinned = true) {
  const size_t tb = p.tiles.size() * sizeof(TileDesc);
  const size_t rb = p.ranges.size() * sizeof(RangeDesc);
  const size_t kb = p.packs.size() * sizeof(PackMask);
  const size_t pb = p.pieces.size() * sizeof(PackPiece);
  char* rbase = base + align256(tb);
  char* kbase = rbase + align256(rb);
  char* pbase = kbase + align256(kb);
  const std::pair<char*, std::pair<const void*, size_t>> parts[] = {
      {base, {p.tiles.data(), tb}}, {rbase, {p.ranges.data(), rb}}, {kbase, {p.packs.data(), kb}},
      {pbase, {p.pieces.data(), pb}}};
  for (const auto& part : parts) {
    const cudaError_t e = h2d_async(part.first, part.second.first, part.second.second, st, pinned);
    if (e != cudaSuccess) return e;
  }
  a.tiles = reinterpret_cast<const TileDesc*>(base);
  a.ranges = reinterpret_cast<const RangeDesc*>(rbase);
  a.packs = kb ? reinterpret_cast<const PackMask*>(kbase) : nullptr;
  a.pieces = pb ? reinterpret_cast<const PackPiece*>(pbase) : nullptr;
  return cudaSuccess;
}

// Debug checks (cp_set_debug_checks): process-wide, read when a call starts.
std::atomic<int32_t> g_debug_checks{0};

// Uploads a plan into the workspace at `base` and points the kernel
// arguments at it.  With debug checks on, every entry is first checked on
// the host against the rows its tensors have (tile_rows for the tiles,
// range_rows for the runs); an inconsistent plan is refused before any GPU
// work of the call.
cp_status_t stage_plan(const Plan& p, char* base, cudaStream_t st, AttnArgs& a, int64_t tile_rows,
                       int64_t range_rows, bool pinned = true) {
  if (a.debug) {
    for (int32_t i = 0; i < int32_t(p.tiles.size()); ++i)
      if (plan_entry_check(p.tiles.data(), int32_t(p.tiles.size()), p.ranges.data(), int32_t(p.ranges.size()),
                           p.packs.data(), int32_t(p.packs.size()), p.pieces.data(), int32_t(p.pieces.size()), i,
                           0, 1, 0, 1, tile_rows, range_rows, a.block_mode, a.lse_stride) != 0)
        return CP_ERR_INVALID_ARG;
  }
  if (upload_plan(p, base, st, a, pinned) != cudaSuccess) return CP_ERR_CUDA;
  a.num_tiles = int32_t(p.tiles.size());
  a.num_ranges = int32_t(p.ranges.size());
  a.num_packs = int32_t(p.packs.size());
  a.num_pieces = int32_t(p.pieces.size());
  a.max_ranges = p.max_ranges;
  return CP_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

bool use_tc_fwd(const cp_desc_t* d) {
  return d->dtype == CP_DT_BF16 && tc_fwd_supported(d->d_qk, d->d_v);
}
bool use_tc_bwd(const cp_desc_t* d) {
  return d->dtype == CP_DT_BF16 && tc_bwd_supported(d->d_qk, d->d_v);
}
// The whole forward's plan and the dQ kernel's: the tensor-core kernels read
// gathered key tiles.
PlanKind fwd_plan_kind(const cp_desc_t* d) { return use_tc_fwd(d) ? kPlanQueryMajorPacked : kPlanQueryMajor; }
PlanKind dq_plan_kind(const cp_desc_t* d) { return use_tc_bwd(d) ? kPlanQueryMajorPacked : kPlanQueryMajor; }
// The dK/dV kernel's: gathered query tiles where its query steps are 128 rows.
PlanKind dkdv_plan_kind(const cp_desc_t* d) {
  return use_tc_bwd(d) && d->d_qk == 128 ? kPlanKeyMajorPacked : kPlanKeyMajor;
}

AttnArgs base_args(const cp_desc_t* d) {
  AttnArgs a{};
  a.T = d->total_tokens;
  a.lse_stride = d->total_tokens;
  a.hq = d->hq;
  a.hkv = d->hkv;
  a.d_qk = d->d_qk;
  a.d_v = d->d_v;
  a.gqa_interleaved = d->gqa == CP_GQA_INTERLEAVED;
  a.causal = d->causal;
  a.scale = d->scale;
  a.debug = g_debug_checks.load();
  return a;
}

// Uploads the key-major plan into `ws` and launches the dK/dV kernel.
cp_status_t run_bwd_dkdv(const cp_desc_t* d, const ShardMap& m, AttnArgs a, char* ws, size_t ws_bytes,
                         cudaStream_t cs) {
  const auto pbp = get_plan(d, m, dkdv_plan_kind(d));
  const Plan& pb = *pbp;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < plan_bytes(pb)) return CP_ERR_WORKSPACE;
  const cp_status_t st = stage_plan(pb, ws, cs, a, d->total_tokens, d->total_tokens);
  if (st != CP_OK) return st;
  const cudaError_t e = use_tc_bwd(d) ? launch_tc_bwd_dkdv(a, cs) : launch_simt_bwd_dkdv(a, d->dtype, cs);
  return e == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

// Uploads the query-major plan into `ws` and launches the dQ kernel.
cp_status_t run_bwd_dq(const cp_desc_t* d, const ShardMap& m, AttnArgs a, char* ws, size_t ws_bytes,
                       cudaStream_t cs) {
  const auto pfp = get_plan(d, m, dq_plan_kind(d));
  const Plan& pf = *pfp;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < plan_bytes(pf)) return CP_ERR_WORKSPACE;
  const cp_status_t st = stage_plan(pf, ws, cs, a, d->total_tokens, d->total_tokens);
  if (st != CP_OK) return st;
  const cudaError_t e = use_tc_bwd(d) ? launch_tc_bwd_dq(a, cs) : launch_simt_bwd_dq(a, d->dtype, cs);
  return e == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

AttnArgs bwd_args(const cp_desc_t* d, const void* q, const void* k, const void* v, const float* lse,
                  const float* dpsum, const void* dout) {
  AttnArgs a = base_args(d);
  a.q = q;
  a.k = k;
  a.v = v;
  a.lse_in = lse;
  a.dpsum = const_cast<float*>(dpsum);
  a.dout = dout;
  return a;
}

struct BwdLayout {
  size_t fwd_plan, bwd_plan, dpsum, total;
};

// ---------------------------------------------------------------- linear attention
// Decayed linear attention has a query head per key/value head (no GQA), a
// causal recurrence, head dims up to 128, and the AllGather CP of the pages
// cuts every sequence into C contiguous pieces.
cp_status_t check_lin(const cp_desc_t* d) {
  cp_status_t st = check_map_fields(d);
  if (st != CP_OK) return st;
  if (d->hq < 1 || d->hkv != d->hq || d->d_qk < 1 || d->d_v < 1) return CP_ERR_INVALID_ARG;
  if (d->dtype != CP_DT_F32 && d->dtype != CP_DT_BF16) return CP_ERR_INVALID_ARG;
  if (!(d->scale > 0.f) || !std::isfinite(d->scale)) return CP_ERR_INVALID_ARG;
  if (d->causal != 1 || d->layout != CP_LAYOUT_CONTIGUOUS) return CP_ERR_UNSUPPORTED;
  if (d->d_qk > 128 || d->d_v > 128 || d->d_qk % 8 || d->d_v % 8) return CP_ERR_UNSUPPORTED;
  return CP_OK;
}

// Blocks of every sequence in order: its rank pieces in rank order, each cut
// into blocks of at most kLinBlock tokens; seq_begin[s] is the first block of
// sequence s (S + 1 entries).
struct LinBlocks {
  std::vector<LinBlock> blocks;
  std::vector<int32_t> seq_begin;
};
LinBlocks lin_blocks(const ShardMap& m) {
  LinBlocks B;
  for (int s = 0; s < m.S; ++s) {
    B.seq_begin.push_back(int32_t(B.blocks.size()));
    for (int r = 0; r < m.C; ++r) {
      const Chunk& c = m.at(r, s, 0);
      for (int32_t o = 0; o < c.len; o += kLinBlock)
        B.blocks.push_back(LinBlock{int32_t(c.srow0 + o), std::min(kLinBlock, c.len - o)});
    }
  }
  B.seq_begin.push_back(int32_t(B.blocks.size()));
  return B;
}

struct LinLayout {
  size_t blocks, seq_begin, states, init, total;
};
LinLayout lin_layout(const cp_desc_t* d, const LinBlocks& B) {
  const size_t st = B.blocks.size() * d->hq * size_t(d->d_qk) * d->d_v * 4;
  LinLayout L{};
  L.blocks = 0;
  L.seq_begin = align256(std::max<size_t>(B.blocks.size(), 1) * sizeof(LinBlock));
  L.states = L.seq_begin + align256(B.seq_begin.size() * 4);
  L.init = L.states + align256(st);
  L.total = L.init + align256(st);
  return L;
}

// ---------------------------------------------------------------- Ulysses
// "Ulysses Context Parallelism 的工程取舍全记录" §1.2 / §2: the all-to-all hands
// rank r heads r*H/C .. (r+1)*H/C - 1 of the whole sequence; with GQA every
// rank needs whole KV heads, so C must divide hq and hkv (blocked GQA keeps a
// rank's query heads on its own KV heads).
cp_status_t check_ulysses(const cp_desc_t* d) {
  const int C = d->cp_size;
  if (d->hq % C != 0 || d->hkv % C != 0) return CP_ERR_UNSUPPORTED;
  if (d->gqa != CP_GQA_BLOCKED && d->hq != d->hkv) return CP_ERR_UNSUPPORTED;
  if (int64_t(C) * d->total_tokens > INT32_MAX) return CP_ERR_UNSUPPORTED;
  return CP_OK;
}

// Global row of every sharded row (the shard map's permutation).
std::vector<int32_t> sharded_to_global(const ShardMap& m, int64_t T) {
  std::vector<int32_t> perm(static_cast<size_t>(T));
  for (const Chunk& c : m.chunks)
    for (int32_t i = 0; i < c.len; ++i) perm[size_t(c.srow0 + i)] = int32_t(c.grow0 + int64_t(i) * c.stride);
  return perm;
}

// The C per-rank unsharded problems as one problem: rank r's block of the
// head-sharded tensors is a copy of the whole sequence set (rows r*T ..),
// with H/C heads; cp_size 1 (full-sequence attention, the pages' "完整
// FlashAttention" per device).
struct UlyssesProblem {
  cp_desc_t u;
  std::vector<int32_t> cu;
};
UlyssesProblem ulysses_problem(const cp_desc_t* d) {
  UlyssesProblem p;
  const std::vector<int32_t> cu = seqlens_of(d);
  const int C = d->cp_size;
  p.cu.push_back(0);
  for (int r = 0; r < C; ++r)
    for (size_t s = 1; s < cu.size(); ++s) p.cu.push_back(int32_t(int64_t(r) * d->total_tokens + cu[s]));
  p.u = *d;
  p.u.total_tokens = int64_t(C) * d->total_tokens;
  p.u.num_seqs = C * (int32_t(cu.size()) - 1);
  p.u.cu_seqlens = p.cu.data();
  p.u.hq = d->hq / C;
  p.u.hkv = d->hkv / C;
  p.u.cp_size = 1;
  p.u.layout = CP_LAYOUT_CONTIGUOUS;
  return p;
}

// Workspace of the Ulysses attention calls: the row map, the head-sharded
// copies of the tensors and the inner call's own workspace.
struct UlyssesLayout {
  size_t perm, q, k, v, o, dout, dq, dk, dv, lse, inner, inner_bytes, total;
};
UlyssesLayout ulysses_layout(const cp_desc_t* d, const cp_desc_t& u, bool bwd) {
  const size_t elt = d->dtype == CP_DT_BF16 ? 2 : 4;
  const size_t T = size_t(d->total_tokens);
  const size_t nq = align256(T * d->hq * d->d_qk * elt), nk = align256(T * d->hkv * d->d_qk * elt);
  const size_t nv = align256(T * d->hkv * d->d_v * elt), no = align256(T * d->hq * d->d_v * elt);
  UlyssesLayout L{};
  size_t off = 0;
  auto take = [&](size_t n) { const size_t at = off; off += n; return at; };
  L.perm = take(align256(T * 4));
  L.q = take(nq);
  L.k = take(nk);
  L.v = take(nv);
  L.o = take(no);
  L.lse = take(align256(T * d->hq * 4));
  if (bwd) {
    L.dout = take(no);
    L.dq = take(nq);
    L.dk = take(nk);
    L.dv = take(nv);
  }
  size_t inner = 0;
  cp_workspace_size(&u, bwd ? CP_OP_BWD : CP_OP_FWD, &inner);
  L.inner = take(align256(inner));
  L.inner_bytes = align256(inner);
  L.total = off;
  return L;
}

BwdLayout bwd_layout(const cp_desc_t* d, const Plan& pf, const Plan& pb) {
  BwdLayout L{};
  L.fwd_plan = 0;
  L.bwd_plan = plan_bytes(pf);
  L.dpsum = L.bwd_plan + plan_bytes(pb);
  L.total = L.dpsum + align256(size_t(d->hq) * size_t(d->total_tokens) * 4);
  return L;
}

// ---------------------------------------------------------------- ring with transport
// Workspace of cp_ring_attn_fwd: the C step plans, two ring buffers of K and
// V (every rank has a slot of slot_rows rows in each), and the fp32 output
// accumulator (bf16 problems; fp32 ones accumulate in o itself).
// The transfers of step s (s = 0 .. C-2) are one copy list per tensor
// (K, then V): every rank's shard into the next rank's slot.  Offsets are
// relative to the list's source (k / v at s = 0, else the step's ring
// buffer) and destination (the other ring buffer).
struct RingLayout {
  std::vector<std::shared_ptr<const Plan>> plans;
  std::vector<size_t> plan_off;
  std::vector<CopySeg> segs;       // all lists, back to back
  std::vector<int32_t> seg_begin;  // list l = 2 * s + tensor: segs[seg_begin[l] .. seg_begin[l + 1])
  std::vector<int64_t> pieces;     // 32 KiB pieces of list l
  int64_t slot_rows = 0;
  size_t segs_off = 0, kslot[2] = {0, 0}, vslot[2] = {0, 0}, oacc = 0, total = 0;
};
RingLayout ring_layout(const cp_desc_t* d, const ShardMap& m) {
  RingLayout L;
  for (int r = 0; r < m.C; ++r) L.slot_rows = std::max<int64_t>(L.slot_rows, m.rank_off[r + 1] - m.rank_off[r]);
  size_t off = 0;
  for (int s = 0; s < m.C; ++s) {
    L.plans.push_back(get_plan(d, m, kPlanQueryMajor, -1, -1, s, L.slot_rows));
    L.plan_off.push_back(off);
    off += plan_bytes(*L.plans.back());
  }
  const size_t elt = d->dtype == CP_DT_BF16 ? 2 : 4;
  const int64_t row_bytes[2] = {int64_t(d->hkv) * d->d_qk * int64_t(elt), int64_t(d->hkv) * d->d_v * int64_t(elt)};
  for (int s = 0; s + 1 < m.C; ++s) {
    for (int t = 0; t < 2; ++t) {
      L.seg_begin.push_back(int32_t(L.segs.size()));
      int64_t pieces = 0;
      for (int r = 0; r < m.C; ++r) {
        const int rho = ((r - s) % m.C + m.C) % m.C;  // the shard rank r holds at step s
        const int64_t rows = m.rank_off[rho + 1] - m.rank_off[rho];
        if (rows == 0) continue;
        CopySeg g;
        g.src = (s == 0 ? m.rank_off[r] : r * L.slot_rows) * row_bytes[t];
        g.dst = int64_t((r + 1) % m.C) * L.slot_rows * row_bytes[t];
        g.bytes = rows * row_bytes[t];
        g.piece0 = pieces;
        pieces += (g.bytes + kPermutePiece - 1) / kPermutePiece;
        L.segs.push_back(g);
      }
      L.pieces.push_back(pieces);
    }
  }
  L.seg_begin.push_back(int32_t(L.segs.size()));
  L.segs_off = off;
  off += align256(std::max<size_t>(L.segs.size(), 1) * sizeof(CopySeg));
  const size_t slot_rows = size_t(m.C) * size_t(L.slot_rows);
  for (int b = 0; b < 2; ++b) {
    L.kslot[b] = off;
    off += align256(slot_rows * d->hkv * d->d_qk * elt);
    L.vslot[b] = off;
    off += align256(slot_rows * d->hkv * d->d_v * elt);
  }
  L.oacc = off;
  if (d->dtype == CP_DT_BF16) off += align256(size_t(d->total_tokens) * d->hq * d->d_v * 4);
  L.total = off;
  return L;
}

}  // namespace
}  // namespace cpattn

// Fixed scratch of cp_attn_fwd_noalloc: the only device memory that entry
// point needs beyond the caller's tensors is the tile plan, kept here.  The
// symbol is a host-side stand-in in host code; its device address is looked
// up once per device below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[CP_NOALLOC_SCRATCH_BYTES];

namespace cpattn {
namespace {

// Device address of g_noalloc_scratch on the current device, looked up on
// the first call for that device (with the device current).
cudaError_t noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* ptrs[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (ptrs[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    ptrs[dev] = p;
  }
  *out = ptrs[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace cpattn

using namespace cpattn;

extern "C" {

const char* cp_status_string(cp_status_t s) {
  switch (s) {
    case CP_OK: return "CP_OK";
    case CP_ERR_INVALID_ARG: return "CP_ERR_INVALID_ARG: invalid descriptor field, pointer or size";
    case CP_ERR_UNSUPPORTED: return "CP_ERR_UNSUPPORTED: valid but not implemented";
    case CP_ERR_CUDA: return "CP_ERR_CUDA: a CUDA runtime call or kernel launch failed";
    case CP_ERR_DEVICE_TIMEOUT: return "CP_ERR_DEVICE_TIMEOUT: a bounded device wait ran out";
    case CP_ERR_WORKSPACE: return "CP_ERR_WORKSPACE: workspace missing, misaligned or too small";
  }
  return "unknown cp_status_t";
}

cp_status_t cp_validate(const cp_desc_t* d) { return check_attn_fields(d); }

cp_status_t cp_workspace_size(const cp_desc_t* d, int32_t op, size_t* bytes) {
  if (bytes == nullptr) return CP_ERR_INVALID_ARG;
  if (op == CP_OP_LIN_FWD) {
    cp_status_t st = check_lin(d);
    if (st != CP_OK) return st;
    *bytes = lin_layout(d, lin_blocks(build_map(d))).total;
    return CP_OK;
  }
  if (op == CP_OP_ULYSSES_A2A) {
    cp_status_t st = check_map_fields(d);
    if (st != CP_OK) return st;
    *bytes = align256(std::max<size_t>(size_t(d->total_tokens), 1) * 4);
    return CP_OK;
  }
  if (op == CP_OP_PERMUTE) {
    cp_status_t st = check_map_fields(d);
    if (st != CP_OK) return st;
    const size_t nseg = d->layout == CP_LAYOUT_STRIPED
                            ? size_t(d->total_tokens)
                            : size_t(d->cp_size) * d->num_seqs * (d->layout == CP_LAYOUT_ZIGZAG ? 2 : 1);
    *bytes = align256(std::max<size_t>(nseg, 1) * sizeof(CopySeg));
    return CP_OK;
  }
  cp_status_t st = check_attn_fields(d);
  if (st != CP_OK) return st;
  ShardMap m = build_map(d);
  if (op == CP_OP_FWD) {
    *bytes = plan_bytes(*get_plan(d, m, fwd_plan_kind(d)));
  } else if (op == CP_OP_BLOCK_FWD) {
    // the largest (q rank, kv rank) plan is bounded by the plan of rank q's
    // tiles against all ranks; size for the worst rank
    size_t mx = 0;
    for (int r = 0; r < m.C; ++r) mx = std::max(mx, plan_bytes(build_fwd_plan(d, m, r, -1)));
    *bytes = mx;
  } else if (op == CP_OP_BWD) {
    *bytes = bwd_layout(d, *get_plan(d, m, dq_plan_kind(d)), *get_plan(d, m, dkdv_plan_kind(d))).total;
  } else if (op == CP_OP_BWD_DKDV) {
    *bytes = plan_bytes(*get_plan(d, m, dkdv_plan_kind(d)));
  } else if (op == CP_OP_BWD_DQ) {
    *bytes = plan_bytes(*get_plan(d, m, dq_plan_kind(d)));
  } else if (op == CP_OP_RING_FWD) {
    *bytes = ring_layout(d, m).total;
  } else if (op == CP_OP_ULYSSES_FWD || op == CP_OP_ULYSSES_BWD) {
    st = check_ulysses(d);
    if (st != CP_OK) return st;
    const UlyssesProblem up = ulysses_problem(d);
    *bytes = ulysses_layout(d, up.u, op == CP_OP_ULYSSES_BWD).total;
  } else {
    return CP_ERR_INVALID_ARG;
  }
  return CP_OK;
}

cp_status_t cp_shard_offsets(const cp_desc_t* d, int64_t* offsets) {
  cp_status_t st = check_map_fields(d);
  if (st != CP_OK) return st;
  if (offsets == nullptr) return CP_ERR_INVALID_ARG;
  ShardMap m = build_map(d);
  for (int r = 0; r <= m.C; ++r) offsets[r] = m.rank_off[r];
  return CP_OK;
}

cp_status_t cp_rank_block_counts(const cp_desc_t* d, int64_t* counts) {
  cp_status_t st = check_attn_fields(d);
  if (st != CP_OK) return st;
  if (counts == nullptr) return CP_ERR_INVALID_ARG;
  ShardMap m = build_map(d);
  const auto pp = get_plan(d, m, kPlanQueryMajor);
  const Plan& p = *pp;
  for (int r = 0; r < m.C; ++r) counts[r] = 0;
  for (const TileDesc& t : p.tiles) counts[t.rank] += t.work;
  return CP_OK;
}

cp_status_t cp_rank_fwd_key_tiles(const cp_desc_t* d, int64_t* counts) {
  cp_status_t st = check_attn_fields(d);
  if (st != CP_OK) return st;
  if (counts == nullptr) return CP_ERR_INVALID_ARG;
  ShardMap m = build_map(d);
  const auto pp = get_plan(d, m, fwd_plan_kind(d));
  for (int r = 0; r < m.C; ++r) counts[r] = 0;
  for (const TileDesc& t : pp->tiles) counts[t.rank] += t.work;
  return CP_OK;
}

cp_status_t cp_shard_permute(const cp_desc_t* d, const void* in, void* out, int64_t row_bytes,
                             int32_t inverse, void* ws, size_t ws_bytes, cp_stream_t stream) {
  CallRange range_("cp_shard_permute");
  cp_status_t st = check_map_fields(d);
  if (st != CP_OK) return st;
  if (row_bytes <= 0 || row_bytes % 16 != 0) return CP_ERR_INVALID_ARG;
  if (inverse != 0 && inverse != 1) return CP_ERR_INVALID_ARG;
  if (d->total_tokens == 0) return CP_OK;
  if (in == nullptr || out == nullptr || !aligned16(in) || !aligned16(out)) return CP_ERR_INVALID_ARG;
  const char* ib = static_cast<const char*>(in);
  const char* ob = static_cast<const char*>(out);
  const int64_t total = d->total_tokens * row_bytes;
  if (ib < ob + total && ob < ib + total) return CP_ERR_INVALID_ARG;  // overlap
  size_t need = 0;
  cp_workspace_size(d, CP_OP_PERMUTE, &need);
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < need) return CP_ERR_WORKSPACE;

  ShardMap m = build_map(d);
  std::vector<CopySeg> segs;
  segs.reserve(m.chunks.size());
  int64_t pieces = 0;
  auto add_seg = [&](int64_t grow, int64_t srow, int64_t rows) {
    CopySeg s;
    const int64_t g = grow * row_bytes, sh = srow * row_bytes;
    s.src = inverse ? sh : g;
    s.dst = inverse ? g : sh;
    s.bytes = rows * row_bytes;
    s.piece0 = pieces;
    pieces += (s.bytes + kPermutePiece - 1) / kPermutePiece;
    segs.push_back(s);
  };
  for (const Chunk& c : m.chunks) {
    if (c.len == 0) continue;
    if (c.stride == 1) {
      add_seg(c.grow0, c.srow0, c.len);
    } else {  // striped: every token is its own segment
      for (int32_t i = 0; i < c.len; ++i) add_seg(c.grow0 + int64_t(i) * c.stride, c.srow0 + i, 1);
    }
  }
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (h2d_async(ws, segs.data(), segs.size() * sizeof(CopySeg), cs) != cudaSuccess) return CP_ERR_CUDA;
  if (launch_permute(static_cast<const CopySeg*>(ws), int32_t(segs.size()), pieces, in, out, cs) !=
      cudaSuccess)
    return CP_ERR_CUDA;
  return CP_OK;
}

cp_status_t cp_lse_merge(const cp_desc_t* d, int64_t rows, float* o_acc, float* lse_acc,
                         const float* o_part, const float* lse_part, cp_stream_t stream) {
  CallRange range_("cp_lse_merge");
  if (d == nullptr || rows < 0) return CP_ERR_INVALID_ARG;
  if (d->hq < 1 || d->d_v < 4 || d->d_v % 4 != 0) return CP_ERR_INVALID_ARG;
  if (rows == 0) return CP_OK;
  if (!o_acc || !lse_acc || !o_part || !lse_part) return CP_ERR_INVALID_ARG;
  if (!aligned16(o_acc) || !aligned16(o_part) || (reinterpret_cast<uintptr_t>(lse_acc) & 3) ||
      (reinterpret_cast<uintptr_t>(lse_part) & 3))
    return CP_ERR_INVALID_ARG;
  if (launch_lse_merge(rows, d->hq, d->d_v, o_acc, lse_acc, o_part, lse_part,
                       reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return CP_ERR_CUDA;
  return CP_OK;
}

cp_status_t cp_attn_block_fwd(const cp_desc_t* d, int32_t q_rank, int32_t kv_rank, const void* q,
                              const void* k, const void* v, float* o_part, float* lse_part, void* ws,
                              size_t ws_bytes, cp_stream_t stream) {
  CallRange range_("cp_attn_block_fwd");
  cp_status_t st = check_attn_fields(d);
  if (st != CP_OK) return st;
  if (q_rank < 0 || q_rank >= d->cp_size || kv_rank < 0 || kv_rank >= d->cp_size)
    return CP_ERR_INVALID_ARG;
  ShardMap m = build_map(d);
  const int64_t Tr = m.rank_off[q_rank + 1] - m.rank_off[q_rank];
  if (Tr == 0) return CP_OK;
  if (!q || !k || !v || !o_part || !lse_part) return CP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o_part) || !aligned16(lse_part))
    return CP_ERR_INVALID_ARG;
  const auto pp = get_plan(d, m, kPlanQueryMajor, q_rank, kv_rank);
  const Plan& p = *pp;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < plan_bytes(p))
    return CP_ERR_WORKSPACE;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  AttnArgs a = base_args(d);
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = o_part;
  a.lse = lse_part;
  a.lse_stride = Tr;
  a.block_mode = 1;
  st = stage_plan(p, static_cast<char*>(ws), cs, a, d->total_tokens, d->total_tokens);
  if (st != CP_OK) return st;
  cudaError_t e = use_tc_fwd(d) ? launch_tc_fwd(a, cs) : launch_simt_fwd(a, d->dtype, cs);
  return e == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

cp_status_t cp_attn_fwd(const cp_desc_t* d, const void* q, const void* k, const void* v, void* o,
                        float* lse, void* ws, size_t ws_bytes, cp_stream_t stream) {
  CallRange range_("cp_attn_fwd");
  cp_status_t st = check_attn_fields(d);
  if (st != CP_OK) return st;
  if (d->total_tokens == 0) return CP_OK;
  if (!q || !k || !v || !o || !lse) return CP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return CP_ERR_INVALID_ARG;
  ShardMap m = build_map(d);
  const auto pp = get_plan(d, m, fwd_plan_kind(d));
  const Plan& p = *pp;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < plan_bytes(p))
    return CP_ERR_WORKSPACE;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  AttnArgs a = base_args(d);
  st = stage_plan(p, static_cast<char*>(ws), cs, a, d->total_tokens, d->total_tokens);
  if (st != CP_OK) return st;
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = o;
  a.lse = lse;
  cudaError_t e = use_tc_fwd(d) ? launch_tc_fwd(a, cs) : launch_simt_fwd(a, d->dtype, cs);
  return e == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

cp_status_t cp_attn_bwd(const cp_desc_t* d, const void* q, const void* k, const void* v,
                        const void* o, const float* lse, const void* dout, void* dq, void* dk,
                        void* dv, void* ws, size_t ws_bytes, cp_stream_t stream) {
  CallRange range_("cp_attn_bwd");
  cp_status_t st = check_attn_fields(d);
  if (st != CP_OK) return st;
  if (d->total_tokens == 0) return CP_OK;
  const void* ptrs[] = {q, k, v, o, lse, dout, dq, dk, dv};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return CP_ERR_INVALID_ARG;
  ShardMap m = build_map(d);
  const auto pfp = get_plan(d, m, dq_plan_kind(d));
  const auto pbp = get_plan(d, m, dkdv_plan_kind(d));
  const Plan& pf = *pfp;
  const Plan& pb = *pbp;
  BwdLayout L = bwd_layout(d, pf, pb);
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < L.total)
    return CP_ERR_WORKSPACE;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(ws);
  float* dpsum = reinterpret_cast<float*>(base + L.dpsum);
  AttnArgs a = bwd_args(d, q, k, v, lse, dpsum, dout);
  a.o = o;
  if (launch_bwd_preprocess(a, d->dtype, cs) != cudaSuccess) return CP_ERR_CUDA;
  AttnArgs ak = a;
  ak.dk = dk;
  ak.dv = dv;
  st = run_bwd_dkdv(d, m, ak, base + L.bwd_plan, L.dpsum - L.bwd_plan, cs);
  if (st != CP_OK) return st;
  AttnArgs aq = a;
  aq.dq = dq;
  return run_bwd_dq(d, m, aq, base + L.fwd_plan, L.bwd_plan - L.fwd_plan, cs);
}

cp_status_t cp_attn_bwd_prep(const cp_desc_t* d, const void* o, const void* dout, float* dpsum, cp_stream_t stream) {
  CallRange range_("cp_attn_bwd_prep");
  cp_status_t st = check_attn_fields(d);
  if (st != CP_OK) return st;
  if (d->total_tokens == 0) return CP_OK;
  if (!o || !dout || !dpsum || !aligned16(o) || !aligned16(dout) || (reinterpret_cast<uintptr_t>(dpsum) & 3))
    return CP_ERR_INVALID_ARG;
  AttnArgs a = base_args(d);
  a.o = o;
  a.dout = dout;
  a.dpsum = dpsum;
  return launch_bwd_preprocess(a, d->dtype, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? CP_OK
                                                                                                 : CP_ERR_CUDA;
}

cp_status_t cp_attn_bwd_dkdv(const cp_desc_t* d, const void* q, const void* k, const void* v, const float* lse,
                             const float* dpsum, const void* dout, void* dk, void* dv, void* ws, size_t ws_bytes,
                             cp_stream_t stream) {
  CallRange range_("cp_attn_bwd_dkdv");
  cp_status_t st = check_attn_fields(d);
  if (st != CP_OK) return st;
  if (d->total_tokens == 0) return CP_OK;
  const void* ptrs[] = {q, k, v, lse, dpsum, dout, dk, dv};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return CP_ERR_INVALID_ARG;
  AttnArgs a = bwd_args(d, q, k, v, lse, dpsum, dout);
  a.dk = dk;
  a.dv = dv;
  return run_bwd_dkdv(d, build_map(d), a, static_cast<char*>(ws), ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

cp_status_t cp_attn_bwd_dq(const cp_desc_t* d, const void* q, const void* k, const void* v, const float* lse,
                           const float* dpsum, const void* dout, void* dq, void* ws, size_t ws_bytes,
                           cp_stream_t stream) {
  CallRange range_("cp_attn_bwd_dq");
  cp_status_t st = check_attn_fields(d);
  if (st != CP_OK) return st;
  if (d->total_tokens == 0) return CP_OK;
  const void* ptrs[] = {q, k, v, lse, dpsum, dout, dq};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return CP_ERR_INVALID_ARG;
  AttnArgs a = bwd_args(d, q, k, v, lse, dpsum, dout);
  a.dq = dq;
  return run_bwd_dq(d, build_map(d), a, static_cast<char*>(ws), ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

cp_status_t cp_attn_fwd_noalloc(const cp_desc_t* d, const void* q, const void* k, const void* v, void* o,
                                float* lse, cp_stream_t stream) {
  cp_status_t st = check_attn_fields(d);
  if (st != CP_OK) return st;
  if (d->total_tokens == 0) return CP_OK;
  ShardMap m = build_map(d);
  const auto pp = get_plan(d, m, fwd_plan_kind(d));
  const Plan& p = *pp;
  if (plan_bytes(p) > CP_NOALLOC_SCRATCH_BYTES) return CP_ERR_WORKSPACE;
  if (!q || !k || !v || !o || !lse) return CP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return CP_ERR_INVALID_ARG;
  void* scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess) return CP_ERR_CUDA;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  AttnArgs a = base_args(d);
  // straight from the cached plan: this entry point allocates nothing, not
  // even the staging ring
  st = stage_plan(p, static_cast<char*>(scratch), cs, a, d->total_tokens, d->total_tokens, false);
  if (st != CP_OK) return st;
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = o;
  a.lse = lse;
  cudaError_t e = use_tc_fwd(d) ? launch_tc_fwd(a, cs) : launch_simt_fwd(a, d->dtype, cs);
  return e == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}

cp_status_t cp_ring_attn_fwd(const cp_desc_t* d, const void* q, const void* k, const void* v, void* o, float* lse,
                             void* ws, size_t ws_bytes, cp_stream_t stream, cp_stream_t comm_stream) {
  CallRange range_("cp_ring_attn_fwd");
  cp_status_t st = check_attn_fields(d);
  if (st != CP_OK) return st;
  if (d->total_tokens == 0) return CP_OK;
  const void* ptrs[] = {q, k, v, o, lse};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return CP_ERR_INVALID_ARG;
  const ShardMap m = build_map(d);
  const RingLayout L = ring_layout(d, m);
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < L.total) return CP_ERR_WORKSPACE;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaStream_t xs = comm_stream ? reinterpret_cast<cudaStream_t>(comm_stream) : cs;
  char* base = static_cast<char*>(ws);
  const bool tc = use_tc_fwd(d);
  float* oacc = d->dtype == CP_DT_BF16 ? reinterpret_cast<float*>(base + L.oacc) : static_cast<float*>(o);

  std::vector<AttnArgs> args(m.C);
  for (int s = 0; s < m.C; ++s) {
    AttnArgs& a = args[s];
    a = base_args(d);
    a.q = q;
    a.k = s == 0 ? k : base + L.kslot[s % 2];
    a.v = s == 0 ? v : base + L.vslot[s % 2];
    a.T_kv = s == 0 ? 0 : int64_t(m.C) * L.slot_rows;
    a.out = oacc;
    a.lse = lse;
    a.lse_stride = d->total_tokens;
    a.block_mode = s == 0 ? 1 : 2;
    st = stage_plan(*L.plans[s], base + L.plan_off[s], cs, a, d->total_tokens, a.T_kv ? a.T_kv : d->total_tokens);
    if (st != CP_OK) return st;
  }
  cudaEvent_t ev_comp = nullptr, ev_comm = nullptr;
  auto cleanup = [&](cp_status_t r) {
    if (ev_comp) cudaEventDestroy(ev_comp);  // released once the recorded work completes
    if (ev_comm) cudaEventDestroy(ev_comm);
    return r;
  };
  if (cudaEventCreateWithFlags(&ev_comp, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&ev_comm, cudaEventDisableTiming) != cudaSuccess)
    return cleanup(CP_ERR_CUDA);
  // A key tile that starts near the end of a shard also loads the slot rows
  // after it.  Their columns are masked (P = 0), but 0 times a stale NaN
  // pattern is NaN, so the ring buffers start out zeroed.
  if (cudaMemsetAsync(base + L.kslot[0], 0, L.oacc - L.kslot[0], cs) != cudaSuccess) return cleanup(CP_ERR_CUDA);
  if (!L.segs.empty() && h2d_async(base + L.segs_off, L.segs.data(), L.segs.size() * sizeof(CopySeg), cs) !=
                             cudaSuccess)
    return cleanup(CP_ERR_CUDA);
  // the inputs (and the uploaded plans) are ready on the compute stream
  if (cudaEventRecord(ev_comp, cs) != cudaSuccess) return cleanup(CP_ERR_CUDA);
  for (int s = 0; s < m.C; ++s) {
    // step s reads the slot the transfer of step s-1 filled
    if (s > 0 && cudaStreamWaitEvent(cs, ev_comm, 0) != cudaSuccess) return cleanup(CP_ERR_CUDA);
    if (s + 1 < m.C) {
      // transport for step s+1, overlapping step s: every rank passes the
      // shard it holds to the next rank.  It overwrites the slots step s-1
      // read, so it waits for that step.
      // One copy kernel per tensor with one CTA per SM: a device-to-device
      // cudaMemcpyAsync runs as a kernel too, and if it is enqueued as the
      // attention kernel starts it takes every SM first; these CTAs fit
      // beside the attention kernel's and copy while it computes.
      if (cudaStreamWaitEvent(xs, ev_comp, 0) != cudaSuccess) return cleanup(CP_ERR_CUDA);
      for (int t = 0; t < 2; ++t) {
        const int l = 2 * s + t;
        const int32_t nseg = L.seg_begin[l + 1] - L.seg_begin[l];
        if (nseg == 0) continue;
        const void* src = s == 0 ? (t == 0 ? k : v) : base + (t == 0 ? L.kslot[s % 2] : L.vslot[s % 2]);
        char* dst = base + (t == 0 ? L.kslot[(s + 1) % 2] : L.vslot[(s + 1) % 2]);
        const CopySeg* segs = reinterpret_cast<const CopySeg*>(base + L.segs_off) + L.seg_begin[l];
        if (launch_permute(segs, nseg, L.pieces[l], src, dst, xs, 1) != cudaSuccess) return cleanup(CP_ERR_CUDA);
      }
      if (cudaEventRecord(ev_comm, xs) != cudaSuccess) return cleanup(CP_ERR_CUDA);
    }
    // block step s: write (s = 0) or merge into (s > 0) the accumulator
    const cudaError_t e = tc ? launch_tc_fwd(args[s], cs) : launch_simt_fwd(args[s], d->dtype, cs);
    if (e != cudaSuccess) return cleanup(CP_ERR_CUDA);
    if (cudaEventRecord(ev_comp, cs) != cudaSuccess) return cleanup(CP_ERR_CUDA);
  }
  if (d->dtype == CP_DT_BF16 &&
      launch_cast_bf16(oacc, o, d->total_tokens * d->hq * int64_t(d->d_v), cs) != cudaSuccess)
    return cleanup(CP_ERR_CUDA);
  return cleanup(CP_OK);
}

cp_status_t cp_ulysses_a2a(const cp_desc_t* d, const void* in, void* out, int32_t heads, int64_t head_bytes,
                           int32_t inverse, void* ws, size_t ws_bytes, cp_stream_t stream) {
  CallRange range_("cp_ulysses_a2a");
  cp_status_t st = check_map_fields(d);
  if (st != CP_OK) return st;
  if (heads < 1 || heads % d->cp_size != 0 || head_bytes <= 0 || head_bytes % 16 != 0) return CP_ERR_INVALID_ARG;
  if (inverse != 0 && inverse != 1) return CP_ERR_INVALID_ARG;
  if (d->total_tokens == 0) return CP_OK;
  if (in == nullptr || out == nullptr || !aligned16(in) || !aligned16(out)) return CP_ERR_INVALID_ARG;
  const int64_t total = d->total_tokens * heads * head_bytes;
  const char* ib = static_cast<const char*>(in);
  const char* ob = static_cast<const char*>(out);
  if (ib < ob + total && ob < ib + total) return CP_ERR_INVALID_ARG;  // overlap
  const size_t need = align256(size_t(d->total_tokens) * 4);
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < need) return CP_ERR_WORKSPACE;
  const std::vector<int32_t> perm = sharded_to_global(build_map(d), d->total_tokens);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (h2d_async(ws, perm.data(), perm.size() * 4, cs) != cudaSuccess) return CP_ERR_CUDA;
  const int64_t chunk = int64_t(heads / d->cp_size) * head_bytes;
  return launch_ulysses_a2a(static_cast<const int32_t*>(ws), d->total_tokens, d->cp_size, chunk, in, out, inverse,
                            cs) == cudaSuccess
             ? CP_OK
             : CP_ERR_CUDA;
}

cp_status_t cp_ulysses_attn_fwd(const cp_desc_t* d, const void* q, const void* k, const void* v, void* o,
                                float* lse, void* ws, size_t ws_bytes, cp_stream_t stream) {
  CallRange range_("cp_ulysses_attn_fwd");
  cp_status_t st = check_attn_fields(d);
  if (st != CP_OK) return st;
  st = check_ulysses(d);
  if (st != CP_OK) return st;
  if (d->total_tokens == 0) return CP_OK;
  const void* ptrs[] = {q, k, v, o, lse};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return CP_ERR_INVALID_ARG;
  const UlyssesProblem up = ulysses_problem(d);
  const UlyssesLayout L = ulysses_layout(d, up.u, false);
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < L.total) return CP_ERR_WORKSPACE;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(ws);
  const int32_t* perm = reinterpret_cast<const int32_t*>(base + L.perm);
  const std::vector<int32_t> hperm = sharded_to_global(build_map(d), d->total_tokens);
  if (h2d_async(base + L.perm, hperm.data(), hperm.size() * 4, cs) != cudaSuccess)
    return CP_ERR_CUDA;
  const int64_t T = d->total_tokens;
  const int C = d->cp_size, elt = d->dtype == CP_DT_BF16 ? 2 : 4;
  // all-to-all #1: sequence shards -> head shards
  if (launch_ulysses_a2a(perm, T, C, int64_t(d->hq / C) * d->d_qk * elt, q, base + L.q, 0, cs) != cudaSuccess ||
      launch_ulysses_a2a(perm, T, C, int64_t(d->hkv / C) * d->d_qk * elt, k, base + L.k, 0, cs) != cudaSuccess ||
      launch_ulysses_a2a(perm, T, C, int64_t(d->hkv / C) * d->d_v * elt, v, base + L.v, 0, cs) != cudaSuccess)
    return CP_ERR_CUDA;
  // full-sequence attention of every rank's heads
  st = cp_attn_fwd(&up.u, base + L.q, base + L.k, base + L.v, base + L.o, reinterpret_cast<float*>(base + L.lse),
                   base + L.inner, L.inner_bytes, stream);
  if (st != CP_OK) return st;
  // all-to-all #2: head shards -> sequence shards
  if (launch_ulysses_a2a(perm, T, C, int64_t(d->hq / C) * d->d_v * elt, base + L.o, o, 1, cs) != cudaSuccess ||
      launch_ulysses_lse(perm, T, C, d->hq, reinterpret_cast<const float*>(base + L.lse), lse, 1, cs) != cudaSuccess)
    return CP_ERR_CUDA;
  return CP_OK;
}

cp_status_t cp_ulysses_attn_bwd(const cp_desc_t* d, const void* q, const void* k, const void* v, const void* o,
                                const float* lse, const void* dout, void* dq, void* dk, void* dv, void* ws,
                                size_t ws_bytes, cp_stream_t stream) {
  CallRange range_("cp_ulysses_attn_bwd");
  cp_status_t st = check_attn_fields(d);
  if (st != CP_OK) return st;
  st = check_ulysses(d);
  if (st != CP_OK) return st;
  if (d->total_tokens == 0) return CP_OK;
  const void* ptrs[] = {q, k, v, o, lse, dout, dq, dk, dv};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return CP_ERR_INVALID_ARG;
  const UlyssesProblem up = ulysses_problem(d);
  const UlyssesLayout L = ulysses_layout(d, up.u, true);
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < L.total) return CP_ERR_WORKSPACE;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(ws);
  const int32_t* perm = reinterpret_cast<const int32_t*>(base + L.perm);
  const std::vector<int32_t> hperm = sharded_to_global(build_map(d), d->total_tokens);
  if (h2d_async(base + L.perm, hperm.data(), hperm.size() * 4, cs) != cudaSuccess)
    return CP_ERR_CUDA;
  const int64_t T = d->total_tokens;
  const int C = d->cp_size, elt = d->dtype == CP_DT_BF16 ? 2 : 4;
  const int64_t cq = int64_t(d->hq / C) * d->d_qk * elt, ck = int64_t(d->hkv / C) * d->d_qk * elt;
  const int64_t cv = int64_t(d->hkv / C) * d->d_v * elt, co = int64_t(d->hq / C) * d->d_v * elt;
  if (launch_ulysses_a2a(perm, T, C, cq, q, base + L.q, 0, cs) != cudaSuccess ||
      launch_ulysses_a2a(perm, T, C, ck, k, base + L.k, 0, cs) != cudaSuccess ||
      launch_ulysses_a2a(perm, T, C, cv, v, base + L.v, 0, cs) != cudaSuccess ||
      launch_ulysses_a2a(perm, T, C, co, o, base + L.o, 0, cs) != cudaSuccess ||
      launch_ulysses_a2a(perm, T, C, co, dout, base + L.dout, 0, cs) != cudaSuccess ||
      launch_ulysses_lse(perm, T, C, d->hq, lse, reinterpret_cast<float*>(base + L.lse), 0, cs) != cudaSuccess)
    return CP_ERR_CUDA;
  st = cp_attn_bwd(&up.u, base + L.q, base + L.k, base + L.v, base + L.o, reinterpret_cast<const float*>(base + L.lse),
                   base + L.dout, base + L.dq, base + L.dk, base + L.dv, base + L.inner, L.inner_bytes, stream);
  if (st != CP_OK) return st;
  if (launch_ulysses_a2a(perm, T, C, cq, base + L.dq, dq, 1, cs) != cudaSuccess ||
      launch_ulysses_a2a(perm, T, C, ck, base + L.dk, dk, 1, cs) != cudaSuccess ||
      launch_ulysses_a2a(perm, T, C, cv, base + L.dv, dv, 1, cs) != cudaSuccess)
    return CP_ERR_CUDA;
  return CP_OK;
}

cp_status_t cp_lin_attn_fwd(const cp_desc_t* d, const void* q, const void* k, const void* v, const float* g, void* o,
                            void* ws, size_t ws_bytes, cp_stream_t stream) {
  CallRange range_("cp_lin_attn_fwd");
  cp_status_t st = check_lin(d);
  if (st != CP_OK) return st;
  if (d->total_tokens == 0) return CP_OK;
  const void* ptrs[] = {q, k, v, g, o};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return CP_ERR_INVALID_ARG;
  const ShardMap m = build_map(d);
  const LinBlocks B = lin_blocks(m);
  const LinLayout L = lin_layout(d, B);
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < L.total) return CP_ERR_WORKSPACE;
  if (B.blocks.empty()) return CP_OK;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(ws);
  if (h2d_async(base + L.blocks, B.blocks.data(), B.blocks.size() * sizeof(LinBlock), cs) != cudaSuccess ||
      h2d_async(base + L.seq_begin, B.seq_begin.data(), B.seq_begin.size() * 4, cs) != cudaSuccess)
    return CP_ERR_CUDA;
  return launch_lin_attn(reinterpret_cast<const LinBlock*>(base + L.blocks), int32_t(B.blocks.size()),
                         reinterpret_cast<const int32_t*>(base + L.seq_begin), m.S, d->hq, d->total_tokens, d->d_qk,
                         d->d_v, d->scale,
                         d->dtype, q, k, v, g, reinterpret_cast<float*>(base + L.states),
                         reinterpret_cast<float*>(base + L.init), o, cs) == cudaSuccess
             ? CP_OK
             : CP_ERR_CUDA;
}

cp_status_t cp_set_debug_checks(int32_t on, int32_t* previous) {
  if (on != 0 && on != 1) return CP_ERR_INVALID_ARG;
  const int32_t old = g_debug_checks.exchange(on);
  if (previous) *previous = old;
  return CP_OK;
}

cp_status_t cp_device_status(cp_stream_t stream, int32_t* code) {
  if (code == nullptr) return CP_ERR_INVALID_ARG;
  if (read_and_clear_device_status(code, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return CP_ERR_CUDA;
  return *code == 0 ? CP_OK : CP_ERR_DEVICE_TIMEOUT;
}

cp_status_t cp_check_bounded_wait(int64_t timeout_ns, int32_t* code, cp_stream_t stream) {
  if (code == nullptr || timeout_ns < 100000 || timeout_ns > 5000000000LL) return CP_ERR_INVALID_ARG;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  int32_t dummy = 0;
  if (read_and_clear_device_status(&dummy, cs) != cudaSuccess) return CP_ERR_CUDA;
  if (launch_wait_selftest(timeout_ns, cs) != cudaSuccess) return CP_ERR_CUDA;
  if (read_and_clear_device_status(code, cs) != cudaSuccess) return CP_ERR_CUDA;
  return CP_OK;
}

}  // extern "C"
