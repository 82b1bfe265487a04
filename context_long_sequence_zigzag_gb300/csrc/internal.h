// internal.h — structures shared by the host runtime and the kernels of
// libcpattn.  Not part of the public ABI (that is include/cp_attn.h).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "cp_attn.h"

namespace cpattn {

// Rows per attention tile on both sides (queries and keys).
constexpr int kTile = 128;

// A tile: up to kTile consecutive SHARDED rows that hold consecutive
// positions of one sequence (tiles never cross a chunk boundary).
// In the forward plan a tile is a query tile and its ranges are key runs; in
// the backward plan a tile is a key tile and its ranges are query runs.
struct TileDesc {
  int32_t row0;         // first sharded row
  int32_t nrows;        // 1..kTile
  int32_t pos0;         // position of row0 inside its sequence
  int32_t range_begin;  // first entry in the range array
  int32_t range_count;  // number of runs this tile visits, in ring order
  int32_t out_row0;     // output row of row0 (block mode: relative to the shard)
  int32_t work;         // number of kTile-row steps over all its runs
  int32_t rank;         // virtual rank that owns the tile
};
static_assert(sizeof(TileDesc) == 32, "TileDesc layout");

// A run: consecutive sharded rows holding consecutive positions of one
// sequence, already clipped to the rows that can be visible to the tile.
struct RangeDesc {
  int32_t row0;   // first sharded row
  int32_t nrows;  // > 0
  int32_t pos0;   // position of row0 inside its sequence
  int32_t flags;  // bit 0: some (tile row, run row) pair is causally masked
};
static_assert(sizeof(RangeDesc) == 16, "RangeDesc layout");

constexpr int32_t kRangeMasked = 1;
// The run is one key tile gathered from pieces of several runs: row0 is its
// first entry in the piece array, flags >> 8 the number of pieces (1 ..
// kTile / 8), pos0 its entry in the key-mask array, nrows kTile.  Every key
// in it is visible to every row of the query tile, so no causal test applies.
// Only the tensor-core forward's own plan has them.
constexpr int32_t kRangePacked = 2;
constexpr int32_t kPackCountShift = 8;

// A key tile gathered from the ragged tails of the unmasked runs that one
// query tile sees (every key of such a run is visible to every row of the
// tile, so its keys may sit anywhere in the tile).  Pieces start at tile rows
// that are multiples of 8 and follow one another up to row kTile.
struct PackMask {
  uint32_t valid[4];  // bit j % 32 of word j / 32: tile row j holds a key
};
static_assert(sizeof(PackMask) == 16, "PackMask layout");

struct PackPiece {
  int32_t src;   // first sharded row loaded
  int32_t dst;   // first tile row, a multiple of 8
  int32_t rows;  // rows loaded: a multiple of 8, dst + rows <= kTile
  int32_t keys;  // the first `keys` of them are keys (1 .. rows); the rest fill the tile, masked
};
static_assert(sizeof(PackPiece) == 16, "PackPiece layout");

// One contiguous copy of the shard permutation (a chunk of one sequence).
struct CopySeg {
  int64_t src;     // byte offset in the source
  int64_t dst;     // byte offset in the destination
  int64_t bytes;   // length in bytes
  int64_t piece0;  // index of the first 32 KiB piece of this segment
};
static_assert(sizeof(CopySeg) == 32, "CopySeg layout");

constexpr int64_t kPermutePiece = 32768;

// Kernel arguments of every attention launch.
struct AttnArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* o;     // forward output (read by the backward)
  const void* dout;
  void* out;         // forward: o (dtype) or o_part (f32, block mode)
  float* lse;        // forward output / backward input, [hq, lse_stride]
  const float* lse_in;
  float* dpsum;      // backward: D = rowsum(dout * o), [hq, T]
  void* dq;
  void* dk;
  void* dv;
  const TileDesc* tiles;
  const RangeDesc* ranges;
  const PackMask* packs;    // key masks of the gathered key tiles (kRangePacked runs), or null
  const PackPiece* pieces;  // their pieces
  int32_t num_tiles;
  int32_t num_ranges;
  int32_t num_packs;
  int32_t num_pieces;
  int32_t max_ranges;  // longest range list of any tile
  int32_t debug;       // nonzero: every CTA checks its plan entry first (plan_check.cuh)
  int32_t* err;        // device error word (set by the launchers)
  int64_t T;
  int64_t T_kv;        // rows of k / v when they live in their own buffer (0: T)
  int64_t lse_stride;  // T, or the shard's row count in block mode
  int32_t hq, hkv, d_qk, d_v;
  int32_t gqa_interleaved;
  int32_t causal;
  // 0: o (dtype) and lse of the whole result; 1: fp32 partial o and lse of
  // one block; 2: merge the block's partial into the fp32 accumulator at
  // out / lse in place (the ring's per-step update)
  int32_t block_mode;
  float scale;
};

// Device error word (bounded waits that ran out), defined in device_status.cu.
enum : int32_t {
  kErrNone = 0,
  kErrWaitTimeoutBase = 0x100,  // | wait site id
};

// ---- launchers (each returns cudaSuccess or the launch error) ----
// ctas_per_sm bounds the grid: 32 for a copy that has the GPU to itself; 1
// for a copy that must run beside a kernel holding every SM (one 256-thread,
// 40-register CTA fits next to an attention CTA).
cudaError_t launch_permute(const CopySeg* segs, int32_t nseg, int64_t npieces,
                           const void* in, void* out, cudaStream_t st, int32_t ctas_per_sm = 32);
// Linear attention with AllGather CP: a block of at most kLinBlock tokens of
// one rank's piece of one sequence; blocks are listed per sequence in order
// (ranks in order, blocks in order inside a rank).
constexpr int32_t kLinBlock = 512;
struct LinBlock {
  int32_t row0;  // first sharded row
  int32_t len;   // tokens
};
size_t lin_output_smem(int32_t Dk, int32_t Dv);
// T = rows of q, k, v, o ([T, H, D] token-major)
cudaError_t launch_lin_attn(const LinBlock* blocks, int32_t nblocks, const int32_t* seq_begin, int32_t S, int32_t H,
                            int64_t T, int32_t Dk, int32_t Dv, float scale, int32_t dtype, const void* q,
                            const void* k, const void* v, const float* g, float* states, float* init, void* o,
                            cudaStream_t st);
// tensor-core block-state and block-output passes (bf16, 128-wide heads)
bool lin_tc_supported(int32_t dtype, int32_t Dk, int32_t Dv);
cudaError_t launch_lin_state_tc(const LinBlock* blocks, int32_t nblocks, int32_t H, int64_t T, const void* k,
                                const void* v, const float* g, float* states, cudaStream_t st);
cudaError_t launch_lin_output_tc(const LinBlock* blocks, int32_t nblocks, int32_t H, int64_t T, float scale,
                                 const void* q, const void* k, const void* v, const float* g, const float* init,
                                 void* o, cudaStream_t st);

// Ulysses re-layout: perm[s] = global row of sharded row s (T entries, device).
cudaError_t launch_ulysses_a2a(const int32_t* perm, int64_t T, int32_t C, int64_t chunk_bytes, const void* in,
                               void* out, int32_t inverse, cudaStream_t st);
cudaError_t launch_ulysses_lse(const int32_t* perm, int64_t T, int32_t C, int32_t H, const float* in, float* out,
                               int32_t inverse, cudaStream_t st);
// o (bf16) = o_acc (fp32) rounded to nearest even, n elements (n % 8 == 0)
cudaError_t launch_cast_bf16(const float* in, void* out, int64_t n, cudaStream_t st);
cudaError_t launch_lse_merge(int64_t rows, int32_t hq, int32_t dv, float* o_acc, float* lse_acc,
                             const float* o_part, const float* lse_part, cudaStream_t st);
cudaError_t launch_simt_fwd(const AttnArgs& a, int32_t dtype, cudaStream_t st);
cudaError_t launch_bwd_preprocess(const AttnArgs& a, int32_t dtype, cudaStream_t st);
cudaError_t launch_simt_bwd_dq(const AttnArgs& a, int32_t dtype, cudaStream_t st);
cudaError_t launch_simt_bwd_dkdv(const AttnArgs& a, int32_t dtype, cudaStream_t st);
cudaError_t launch_tc_fwd(const AttnArgs& a, cudaStream_t st);
// tensor-core backward: dK/dV over the key-major plan, dQ over the query-major plan
cudaError_t launch_tc_bwd_dkdv(const AttnArgs& a, cudaStream_t st);
cudaError_t launch_tc_bwd_dq(const AttnArgs& a, cudaStream_t st);
bool tc_fwd_supported(int32_t d_qk, int32_t d_v);
bool tc_bwd_supported(int32_t d_qk, int32_t d_v);
cudaError_t read_and_clear_device_status(int32_t* code, cudaStream_t st);
// Device address of the error word on the current device (cached per device).
int32_t* device_error_word();
cudaError_t launch_wait_selftest(int64_t timeout_ns, cudaStream_t st);

}  // namespace cpattn
