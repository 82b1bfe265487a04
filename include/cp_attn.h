/*
 * cp_attn.h — C ABI of libcpattn: context-parallel exact causal attention on
 * one GB300 (sm_103a).
 *
 * A sequence (or a pack of sequences) of T tokens is cut into C context-
 * parallel shards.  The C "virtual ranks" all live on one GPU: the KV ring of
 * ring attention is the order in which the kernels visit the KV shards that
 * are already resident in device memory.  Sources for the method:
 *   - "超长序列并行训练技术：Ulysses与Ring-Attention详解" (Ulysses and Ring-
 *     Attention explained), §4.1 (blockwise attention: each (Q block, KV
 *     block) step yields a partial output and its log-sum-exp, merged by an
 *     update step), §4.2 (the lse merge formula; zigzag pairing of block i
 *     with block 2C-1-i), §4.3 (the backward recomputes instead of storing).
 *   - "超长上下文训练速度翻倍秘籍" (Ling long-context speed-up), §2 pitfall 1
 *     (the local diagonal block is causal, KV blocks of earlier shards are
 *     fully visible), §3 varlen CP (each packed sub-sequence is cut into CP
 *     pieces, described by cu_seqlens).
 *   - "LLM context parallel production guide" (oh-bug.com), sections
 *     "核心原理" (exact merge through softmax statistics), "因果 Attention 会
 *     制造 Rank 负载不均" (skip blocks above the diagonal; zigzag or striped
 *     placement balances the ranks; count effective QK blocks per rank),
 *     "变长序列" and
 *     "位置编码必须跟序列分片一起走" (all position metadata follows the shard map).
 *
 * Conventions shared by every entry point
 *   - Ownership: the caller owns every buffer; the library allocates no
 *     device memory.  Device buffers are plain device pointers; the host
 *     pointers are read during the call only.  For its host-to-device copies
 *     of tile plans and index tables the library keeps one pinned host
 *     staging buffer of 32 MiB per device, allocated by the first call on
 *     that device that needs it and held until the process exits, so that a
 *     call does not wait for earlier work on its stream (cp_attn_fwd_noalloc
 *     never uses it).
 *   - Tracing: every entry point that enqueues GPU work (but
 *     cp_attn_fwd_noalloc) opens an NVTX range named after itself for its
 *     duration on the host, so that a profiler's timeline attributes the
 *     kernels to the call; without a profiler attached this costs nothing.
 *   - Streams: all GPU work is enqueued asynchronously on `stream` (a
 *     cudaStream_t; NULL = the legacy default stream).  A call returns after
 *     enqueueing; errors found on the host are returned before anything is
 *     enqueued.  A status of CP_ERR_CUDA means a CUDA runtime call or a kernel
 *     launch failed (cudaGetLastError is left as the runtime set it).
 *   - Token order: every token-major tensor passed to the attention calls is in
 *     SHARDED order: the concatenation of the C ranks' local buffers, rank 0
 *     first.  cu_seqlens is always given in GLOBAL order; the library derives
 *     the shard map from it.  cp_shard_permute converts between the orders.
 *   - Shard map: sequence s of length L is cut into n pieces at floor(j*L/n),
 *     j = 0..n (pieces differ by at most one token and may be empty).
 *     CONTIGUOUS: n = C, rank r holds piece r.  ZIGZAG: n = 2C, rank r holds
 *     piece r then piece 2C-1-r.  STRIPED: rank r holds the tokens at
 *     positions p with p mod C == r, in increasing position ("LLM context
 *     parallel production guide", 因果 Attention 会制造 Rank 负载不均:
 *     striped token placement; one-token stripes).  Inside a rank, sequences
 *     appear in order.
 *   - Layouts (row-major, innermost last):
 *       q [T, hq, d_qk]   k [T, hkv, d_qk]   v [T, hkv, d_v]
 *       o, dout [T, hq, d_v]   dq [T, hq, d_qk]   dk [T, hkv, d_qk]   dv [T, hkv, d_v]
 *       lse [hq, T] float32, natural log of the sum of exp(scale * q.k) over the
 *       visible keys.  Element type of q/k/v/o/dout/dq/dk/dv = desc.dtype.
 *   - Alignment: every tensor pointer must be 16-byte aligned and
 *     d_qk * elt and d_v * elt must be multiples of 16 bytes.
 *   - Visibility: key j is visible to query i iff they belong to the same
 *     sequence and (causal == 0 or pos(j) <= pos(i)).  A query that sees no key
 *     gets o = 0 and lse = -inf.
 *   - GQA: hq % hkv == 0, G = hq / hkv.  BLOCKED: kv(h) = h / G.
 *     INTERLEAVED: kv(h) = h % hkv.
 *   - Precision: BF16 inputs run on the tcgen05 tensor cores with FP32
 *     accumulation (d_qk in {128, 192}, d_v = 128); other head dims and FP32
 *     inputs run on a CUDA-core FP32 path.  Outputs o/dq/dk/dv are rounded to
 *     desc.dtype (round to nearest even); lse, partial outputs and the merge
 *     are FP32.
 */
#ifndef CP_ATTN_H
#define CP_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here so that this header needs no CUDA
 * header. */
typedef struct CUstream_st* cp_stream_t;

typedef enum {
  CP_OK = 0,
  CP_ERR_INVALID_ARG = 1,    /* a descriptor field, pointer or size is invalid   */
  CP_ERR_UNSUPPORTED = 2,    /* valid but not implemented (e.g. head dim)        */
  CP_ERR_CUDA = 3,           /* a CUDA runtime call or kernel launch failed      */
  CP_ERR_DEVICE_TIMEOUT = 4, /* a kernel's bounded wait ran out (see cp_device_status) */
  CP_ERR_WORKSPACE = 5       /* workspace pointer NULL/misaligned or too small   */
} cp_status_t;

typedef enum { CP_LAYOUT_CONTIGUOUS = 0, CP_LAYOUT_ZIGZAG = 1, CP_LAYOUT_STRIPED = 2 } cp_layout_t;
typedef enum { CP_DT_F32 = 0, CP_DT_BF16 = 1 } cp_dtype_t;
typedef enum { CP_GQA_BLOCKED = 0, CP_GQA_INTERLEAVED = 1 } cp_gqa_t;
typedef enum {
  CP_OP_FWD = 0, CP_OP_BWD = 1, CP_OP_BLOCK_FWD = 2, CP_OP_PERMUTE = 3, CP_OP_BWD_DKDV = 4, CP_OP_BWD_DQ = 5,
  CP_OP_ULYSSES_A2A = 6, CP_OP_ULYSSES_FWD = 7, CP_OP_ULYSSES_BWD = 8, CP_OP_LIN_FWD = 9, CP_OP_RING_FWD = 10
} cp_op_t;

/* Problem descriptor.  Read on the host during each call; not retained. */
typedef struct {
  int64_t total_tokens;       /* T >= 0                                            */
  int32_t num_seqs;           /* >= 1 packed sequences                             */
  int32_t hq, hkv;            /* query heads, key/value heads (hq % hkv == 0)      */
  const int32_t* cu_seqlens;  /* HOST, num_seqs+1 entries, global order: cu[0] = 0,
                                 non-decreasing, cu[num_seqs] = T.  NULL is allowed
                                 only with num_seqs == 1 (one sequence of T).      */
  int32_t d_qk, d_v;          /* head dims of q/k and v/o                          */
  int32_t cp_size;            /* C >= 1 virtual ranks                              */
  int32_t layout;             /* cp_layout_t                                       */
  int32_t causal;             /* 1: causal inside each sequence, 0: full           */
  float scale;                /* softmax scale applied to q.k (> 0, finite)        */
  int32_t gqa;                /* cp_gqa_t                                          */
  int32_t dtype;              /* cp_dtype_t of q/k/v/o/dout/dq/dk/dv               */
} cp_desc_t;

/* Human-readable name of a status code (static string, never NULL). */
const char* cp_status_string(cp_status_t status);

/* Check a descriptor on the host (no GPU work).  Returns CP_OK,
 * CP_ERR_INVALID_ARG or CP_ERR_UNSUPPORTED. */
cp_status_t cp_validate(const cp_desc_t* desc);

/* Workspace bytes needed by one call of operation `op` (cp_op_t) for this
 * descriptor.  Host only.  The workspace must be device memory, 256-byte
 * aligned, at least this large, and must not be used by anything else while
 * the call's kernels run. */
cp_status_t cp_workspace_size(const cp_desc_t* desc, int32_t op, size_t* bytes);

/* Start row of every rank's shard in sharded order: offsets[0..C], host
 * array of C+1 int64 (offsets[C] = T).  Host only. */
cp_status_t cp_shard_offsets(const cp_desc_t* desc, int64_t* offsets);

/* Effective attention work per virtual rank: the number of visible
 * (128-query x 128-key) tiles that rank's queries touch for one head, host
 * array of C int64.  "LLM context parallel production guide", 因果 Attention
 * 会制造 Rank 负载不均: monitor effective QK blocks per rank, not tokens.
 * Key tiles are counted as cut from each run (the bf16 tensor-core forward
 * and dQ kernels may run fewer: they gather the ragged tails of a query
 * tile's unmasked runs into shared key tiles).  Host only. */
cp_status_t cp_rank_block_counts(const cp_desc_t* desc, int64_t* counts);

/* Key tiles the forward (cp_attn_fwd) runs per virtual rank for one head,
 * host array of C int64; the dQ pass of the backward runs the same.  With
 * the bf16 tensor-core kernels this is cp_rank_block_counts less the tiles
 * saved by gathering the ragged tails of each query tile's fully visible
 * runs into shared key tiles (pieces from 8-row boundaries, split across two
 * tiles where one fills); otherwise it equals cp_rank_block_counts.
 * Host only. */
cp_status_t cp_rank_fwd_key_tiles(const cp_desc_t* desc, int64_t* counts);

/* Bit-exact row permutation between global and sharded order
 * ("Ulysses与Ring-Attention详解" §4.2 zigzag table; "LLM context parallel
 * production guide", 位置编码必须跟序列分片一起走: every token-major tensor —
 * q, k, v, positions, masks, labels — follows the same map).
 *   in, out    : device, T rows of row_bytes bytes each; must not overlap
 *   row_bytes  : > 0, multiple of 16; in/out 16-byte aligned
 *   inverse    : 0 = global -> sharded, 1 = sharded -> global
 *   workspace  : cp_workspace_size(desc, CP_OP_PERMUTE) bytes
 * Only total_tokens, num_seqs, cu_seqlens, cp_size and layout are read. */
cp_status_t cp_shard_permute(const cp_desc_t* desc, const void* in, void* out,
                             int64_t row_bytes, int32_t inverse,
                             void* workspace, size_t workspace_bytes, cp_stream_t stream);

/* One ring step: the queries of rank q_rank against the keys/values held by
 * rank kv_rank ("Ulysses与Ring-Attention详解" §4.1 compute_block -> (out, lse);
 * "超长上下文训练速度翻倍秘籍" §2: the q_rank == kv_rank block is causal, keys of
 * earlier positions are fully visible, later ones are skipped).
 *   q, k, v   : full sharded tensors; only the two ranks' rows are read
 *   o_part    : device float32 [T_r, hq, d_v], T_r = rows of rank q_rank;
 *               normalised over the visible keys of this block
 *   lse_part  : device float32 [hq, T_r]; -inf (with o_part = 0) for rows that
 *               see no key of this block
 *   workspace : cp_workspace_size(desc, CP_OP_BLOCK_FWD) bytes */
cp_status_t cp_attn_block_fwd(const cp_desc_t* desc, int32_t q_rank, int32_t kv_rank,
                              const void* q, const void* k, const void* v,
                              float* o_part, float* lse_part,
                              void* workspace, size_t workspace_bytes, cp_stream_t stream);

/* In-place exact merge of a partial result into an accumulator
 * ("Ulysses与Ring-Attention详解" §4.2: lse = log(exp(lse_acc) + exp(lse_part));
 * o = exp(lse_acc - lse) o_acc + exp(lse_part - lse) o_part).  -inf is the
 * identity (an empty partial leaves the accumulator unchanged).
 *   rows      : number of token rows (e.g. T_r of one rank)
 *   o_acc, o_part     : device float32 [rows, hq, d_v]
 *   lse_acc, lse_part : device float32 [hq, rows]
 * Only hq and d_v (multiple of 4) are read from desc. */
cp_status_t cp_lse_merge(const cp_desc_t* desc, int64_t rows,
                         float* o_acc, float* lse_acc,
                         const float* o_part, const float* lse_part, cp_stream_t stream);

/* Fused forward over all ranks: for every rank's queries, the KV shards are
 * visited in ring order r, r-1, ..., r-C+1 (mod C) with the merge done on
 * chip; fully masked tiles are skipped.
 *   q, k, v   : device, sharded order
 *   o         : device [T, hq, d_v] (desc.dtype)
 *   lse       : device float32 [hq, T] (kept for the backward)
 *   workspace : cp_workspace_size(desc, CP_OP_FWD) bytes */
cp_status_t cp_attn_fwd(const cp_desc_t* desc, const void* q, const void* k, const void* v,
                        void* o, float* lse,
                        void* workspace, size_t workspace_bytes, cp_stream_t stream);

/* Backward ("Ulysses与Ring-Attention详解" §4.3): recomputes the attention
 * probabilities from q, k and the stored final lse, with D = rowsum(dout * o),
 * and writes dq, dk, dv (dk/dv summed over the query heads of each GQA group).
 *   o, lse    : outputs of cp_attn_fwd for the same inputs
 *   dout      : device [T, hq, d_v]
 *   dq, dk, dv: device, sharded order, desc.dtype
 *   workspace : cp_workspace_size(desc, CP_OP_BWD) bytes */
cp_status_t cp_attn_bwd(const cp_desc_t* desc, const void* q, const void* k, const void* v,
                        const void* o, const float* lse, const void* dout,
                        void* dq, void* dk, void* dv,
                        void* workspace, size_t workspace_bytes, cp_stream_t stream);

/* Ring attention forward with the KV transport made explicit
 * ("Ulysses Context Parallelism 的工程取舍全记录" §2: ring attention passes
 * the KV blocks rank to rank by point-to-point transfers that overlap the
 * block computation; "LLM context parallel production guide", Ring
 * Attention: every rank computes its local block while the next KV block is
 * in flight; "Ulysses与Ring-Attention详解" §4.1-§4.2: each step's (out, lse)
 * is merged into the running result).
 * Every virtual rank r owns a receive slot in each of two ring buffers.  In
 * step s (s = 0 .. C-1) rank r computes its queries against the shard it
 * holds, rho = (r - s) mod C (its own shard at s = 0, read from k / v; from
 * s = 1 on the copy in its slot), and merges the block's partial into the
 * fp32 accumulator in the kernel's epilogue.  Meanwhile, on comm_stream,
 * every rank sends the shard it holds to rank r + 1 (mod C): its K rows and
 * its V rows are copied into the other ring buffer, which is what a
 * point-to-point transfer between two GPUs becomes when all ranks share one.
 * The copies of a step run as one copy kernel per tensor with a single
 * small CTA per SM, sized to fit beside the attention kernel's CTAs, so
 * that they proceed while it computes (a device-to-device cudaMemcpyAsync is
 * itself a kernel, and launched as the attention kernel starts it takes
 * every SM first).  Give comm_stream a higher priority than stream.  Events
 * order the two streams: step s + 1 waits for the transfer that filled its
 * slots, and that transfer waits for step s - 1, the last reader of the
 * buffer it overwrites.
 *   q, k, v    : device, sharded order (as cp_attn_fwd)
 *   o, lse     : device, as cp_attn_fwd; lse is also the running accumulator
 *   workspace  : cp_workspace_size(desc, CP_OP_RING_FWD) bytes: the C step
 *                plans, the copy lists of the transfers, 2 x 2 ring buffers
 *                of C x max_rank_rows rows of K and of V, and (bf16 problems)
 *                the fp32 o accumulator
 *                [T, hq, d_v]; fp32 problems accumulate in o itself
 *   stream     : compute stream; the call's results are complete when the
 *                work enqueued on it is (the transfers are ordered before the
 *                last step)
 *   comm_stream: stream of the transfers; NULL runs them on `stream` too
 *                (serialised, no overlap)
 * The result equals cp_attn_fwd's up to the rounding order of the merge.
 * The call creates two CUDA events and releases them before it returns
 * (the driver frees them once the enqueued work has used them). */
cp_status_t cp_ring_attn_fwd(const cp_desc_t* desc, const void* q, const void* k, const void* v,
                             void* o, float* lse, void* workspace, size_t workspace_bytes,
                             cp_stream_t stream, cp_stream_t comm_stream);

/* ---------------------------------------------------------------- Ulysses
 * All-to-all ("Ulysses") context parallelism with the C virtual ranks on one
 * GPU ("Ulysses Context Parallelism 的工程取舍全记录" §1.2: before attention an
 * all-to-all turns sequence shards of every head into the whole sequence of
 * H/C heads per device, device r taking heads r*H/C .. (r+1)*H/C - 1; after
 * attention a second all-to-all turns the output back; §2: with GQA every
 * device needs whole KV heads, so C must divide hq and hkv;
 * "超长上下文训练速度翻倍秘籍", All2All CP 实现).  On one GPU the all-to-all is
 * a re-layout between
 *   sharded   [T, H, e] in sharded token order (the layout of every other call), and
 *   head-sharded [C, T, H/C, e]: rank r's block holds heads r*H/C.. of all T
 *                tokens in GLOBAL token order (cu_seqlens order).
 * e = bytes per head (head_bytes). */

/* The all-to-all re-layout, bit-exact.
 *   in, out    : device, T * heads * head_bytes bytes each, 16-byte aligned,
 *                not overlapping
 *   heads      : heads of this tensor (hq for q/o/dq, hkv for k/v/dk/dv);
 *                must be a multiple of cp_size
 *   head_bytes : bytes per head, > 0, multiple of 16
 *   inverse    : 0 = sharded -> head-sharded, 1 = head-sharded -> sharded
 *   workspace  : cp_workspace_size(desc, CP_OP_ULYSSES_A2A) bytes (the row map)
 * Only total_tokens, num_seqs, cu_seqlens, cp_size and layout are read. */
cp_status_t cp_ulysses_a2a(const cp_desc_t* desc, const void* in, void* out, int32_t heads,
                           int64_t head_bytes, int32_t inverse,
                           void* workspace, size_t workspace_bytes, cp_stream_t stream);

/* Ulysses attention forward: the same inputs and outputs as cp_attn_fwd
 * (sharded order, all heads), computed as all-to-all, full-sequence
 * attention of every rank's heads (the tcgen05 kernels with one rank), and
 * all-to-all back.  Results equal cp_attn_fwd's up to rounding order.
 *   workspace : cp_workspace_size(desc, CP_OP_ULYSSES_FWD) bytes; holds the
 *               head-sharded copies of q, k, v, o, lse and the inner plan.
 * CP_ERR_UNSUPPORTED when cp_size does not divide hq and hkv, or with
 * interleaved GQA (hq != hkv). */
cp_status_t cp_ulysses_attn_fwd(const cp_desc_t* desc, const void* q, const void* k, const void* v,
                                void* o, float* lse,
                                void* workspace, size_t workspace_bytes, cp_stream_t stream);

/* Ulysses attention backward: the inputs and outputs of cp_attn_bwd, computed
 * on the head-sharded layout (six re-layouts in, three out).
 *   workspace : cp_workspace_size(desc, CP_OP_ULYSSES_BWD) bytes. */
cp_status_t cp_ulysses_attn_bwd(const cp_desc_t* desc, const void* q, const void* k, const void* v,
                                const void* o, const float* lse, const void* dout,
                                void* dq, void* dk, void* dv,
                                void* workspace, size_t workspace_bytes, cp_stream_t stream);

/* ------------------------------------------------------ linear attention
 * Decayed linear attention with AllGather context parallelism
 * ("超长上下文训练速度翻倍秘籍": per head h_t = alpha h_{t-1} + k_t^T v_t and
 * o_t = scale q_t h_t inside each sequence, alpha = exp(g[head]); AllGather
 * CP: every rank computes the hidden state of its piece from a zero start,
 * the gathered states give each rank its initial state through the prefix
 * kv_state = kv_state * alpha^len + cur over the preceding ranks, and the
 * rank's output is its local output plus (q * alpha^(j+1)) @ init_state for
 * its j-th token).  The output equals the unsharded recurrence.
 *   desc      : hq == hkv heads, d_qk (keys/queries) and d_v up to 128,
 *               causal == 1, layout CONTIGUOUS (pieces cut at floor(r*L/C)),
 *               dtype bf16 or fp32; scale multiplies q
 *   q, k      : device [T, hq, d_qk], v / o: device [T, hq, d_v], sharded order
 *   g         : device float32 [hq], the log of the per-head decay alpha
 *   workspace : cp_workspace_size(desc, CP_OP_LIN_FWD) bytes: the block list
 *               and the gathered local and recovered initial states (fp32
 *               [blocks, hq, d_qk, d_v]; every rank piece is cut into blocks of
 *               at most 512 tokens, the unit of parallel work, and the prefix
 *               runs over the blocks of a sequence in order — ranks in order,
 *               blocks in order inside a rank)
 * bf16 with d_qk == d_v == 128 runs the block states and block outputs as
 * tcgen05 MMAs in chunks of 128 tokens, with fp32 accumulation and the
 * carried state in fp32.  The decayed score matrix, the decay-weighted keys
 * and the state are rounded to bf16 as MMA operands.  Every other shape runs
 * FP32 arithmetic on the CUDA cores.  CP_ERR_UNSUPPORTED for another layout,
 * non-causal, or head dims above 128 or not multiples of 8. */
cp_status_t cp_lin_attn_fwd(const cp_desc_t* desc, const void* q, const void* k, const void* v,
                            const float* g, void* o,
                            void* workspace, size_t workspace_bytes, cp_stream_t stream);

/* Forward without a workspace, for callers that cannot allocate device
 * memory.  The source pages have no counterpart to this entry point.
 *
 * Some callers cannot call cudaMalloc (or any allocator): a plugin whose host
 * framework owns every device allocation and hands it only its input and
 * output tensors, or code on a path where allocating is not allowed.  This
 * variant computes exactly what cp_attn_fwd computes, with the same arguments
 * minus the workspace: its only scratch, the tile plan, lives in a
 * fixed-size array inside the library's device image (CP_NOALLOC_SCRATCH_BYTES
 * = 4 MiB, held by every GPU that loads the library until the process
 * exits).  It calls no cudaMalloc, cudaFree or allocating routine.
 *   - The first call on a device looks up the array's device address (once
 *     per device, on the current device).
 *   - A problem whose plan needs more than CP_NOALLOC_SCRATCH_BYTES is
 *     rejected with CP_ERR_WORKSPACE before any GPU work is enqueued.
 *   - Every call shares the one array and overwrites it with its own plan:
 *     calls whose GPU work overlaps in time (different streams without
 *     ordering) race on it.  Order such calls on one stream or with events. */
#define CP_NOALLOC_SCRATCH_BYTES (4u << 20)
cp_status_t cp_attn_fwd_noalloc(const cp_desc_t* desc, const void* q, const void* k, const void* v,
                                void* o, float* lse, cp_stream_t stream);

/* The backward in three independent pieces (cp_attn_bwd runs all three).
 *
 * cp_attn_bwd_prep: D = rowsum(dout * o) for every (head, row), the second
 * statistic the recomputed backward needs besides lse
 * ("Ulysses与Ring-Attention详解" §4.3).
 *   o, dout : device [T, hq, d_v] (desc.dtype), sharded order
 *   dpsum   : device float32 [hq, T]
 * No workspace. */
cp_status_t cp_attn_bwd_prep(const cp_desc_t* desc, const void* o, const void* dout, float* dpsum,
                             cp_stream_t stream);

/* cp_attn_bwd_dkdv: dk and dv (each summed over the query heads of its GQA
 * group) from q, k, v, the forward's lse, dpsum (cp_attn_bwd_prep) and dout.
 * Key-tile-major: every key tile visits the query runs of all virtual ranks
 * that see it.  workspace: cp_workspace_size(desc, CP_OP_BWD_DKDV) bytes. */
cp_status_t cp_attn_bwd_dkdv(const cp_desc_t* desc, const void* q, const void* k, const void* v,
                             const float* lse, const float* dpsum, const void* dout, void* dk, void* dv,
                             void* workspace, size_t workspace_bytes, cp_stream_t stream);

/* cp_attn_bwd_dq: dq from the same inputs, query-tile-major (dq accumulates
 * on chip over every visible key tile and is written once).
 * workspace: cp_workspace_size(desc, CP_OP_BWD_DQ) bytes.  Independent of
 * cp_attn_bwd_dkdv: the two may run concurrently on different streams, each
 * with its own workspace. */
cp_status_t cp_attn_bwd_dq(const cp_desc_t* desc, const void* q, const void* k, const void* v,
                           const float* lse, const float* dpsum, const void* dout, void* dq,
                           void* workspace, size_t workspace_bytes, cp_stream_t stream);

/* Debug checks, process-wide, for the calls that start after this one
 * (on = 1) or none (on = 0, the default); *previous (may be NULL) receives
 * the former setting.  With checks on, the host checks every tile plan
 * against the row counts of the tensors it indexes before uploading it
 * (CP_ERR_INVALID_ARG if inconsistent), and every CTA of the attention
 * kernels checks its own plan entry (tile index, heads, tile rows, output
 * rows, run list and run rows, step count) before any load or store: a bad
 * entry records 0x200 | check in the device error word (cp_device_status)
 * and the CTA returns without touching memory.  No check traps.  It stands
 * in for a memory checker: the pages report a block-write / scalar-read
 * race that unit tests had missed ("超长上下文训练速度翻倍秘籍" §2). */
cp_status_t cp_set_debug_checks(int32_t on, int32_t* previous);

/* Synchronises `stream`, then returns and clears the device error word of
 * the current device: *code = 0 when every bounded wait since the last call
 * completed, otherwise a nonzero code naming the wait that ran out (and the
 * status CP_ERR_DEVICE_TIMEOUT). */
cp_status_t cp_device_status(cp_stream_t stream, int32_t* code);

/* Self-check of the bounded-wait machinery: launches one kernel that waits
 * on a barrier nothing ever completes, with a limit of timeout_ns
 * nanoseconds (1e5 .. 5e9), and reports through *code what the kernel saw
 * (expected: the timeout code).  Synchronises `stream`.  Leaves the device
 * error word cleared. */
cp_status_t cp_check_bounded_wait(int64_t timeout_ns, int32_t* code, cp_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CP_ATTN_H */
