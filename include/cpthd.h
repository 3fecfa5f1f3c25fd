/*
 * cpthd.h -- C ABI of libcpthd.so: context-parallel causal self-attention over
 * THD-packed documents, every context-parallel (CP) rank emulated on one GPU.
 *
 * Sources of the operations (TransformerEngine pages):
 *   [AG]  "[PyTorch] Add no-load-balance THD all-gather CP"
 *   [A2A] "[PyTorch] Extend no-load-balance CP to the a2a comm type"
 *   [P2P] "THD P2P context-parallel regression when padded cu_seqlens are
 *          value-equal but not object-identical"
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layout "THD": a packed tensor [rows, H, D] of bf16, row-major, one row per
 *   token (row_bytes = 2*H*D).  Documents are delimited by
 *   cu_seqlens_padded ("cup", int32 [n_docs+1], physical offsets, cup[0]=0,
 *   cup[n_docs] = total_tokens = T).  cu_seqlens ("cu", int32 [n_docs+1])
 *   gives the real token counts L_i = cu[i+1]-cu[i] <= P_i = cup[i+1]-cup[i];
 *   document i's real tokens are rows [cup[i], cup[i]+L_i), the rest of its
 *   padded range is padding.  When pad_between_seqs == 0, cu is not read and
 *   L_i = P_i.
 * Strategies ([AG] §What changed, §Why; [A2A] first paragraph):
 *   DUAL_CHUNK_SWAP: each document's padded range is cut into 2*cp_size equal
 *     chunks; rank r holds chunk r then chunk 2*cp_size-1-r of every document,
 *     documents in order.  Needs P_i % (2*cp_size) == 0 for every document.
 *   NO_LOAD_BALANCE: rank r holds the contiguous physical rows
 *     [r*s_local, (r+1)*s_local), s_local = T/cp_size.  Needs T % cp_size == 0.
 *   Both: causal self-attention without a sliding window, equal Q/K/V lengths
 *   ([AG] §Scope and constraints).  Forward and backward must use the same
 *   strategy and the same metadata ([AG] §What changed, 4th item).
 * Memory: the caller owns every buffer (host and device) and the stream.  No
 *   entry point allocates or frees memory or synchronises, except
 *   cp_device_status (documented below).  Device pointers must be 16-byte
 *   aligned.  All launches are asynchronous on `stream` (a cudaStream_t; NULL
 *   is the legacy default stream).
 * Errors: every entry point returns a cp_status_t.  Arguments are validated on
 *   the host before anything is launched; a failed validation launches
 *   nothing.  A failed launch returns CP_ERR_CUDA.  Errors that only the
 *   device can see (bad cu_seqlens values, an out-of-range index) are written
 *   to the metadata header (status field) and to a per-device status word that
 *   cp_device_status reads; kernels given metadata with a non-zero status
 *   write nothing.  Nothing traps the GPU.
 */
#ifndef CPTHD_H
#define CPTHD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CP_DUAL_CHUNK_SWAP = 0, /* default of [AG] */
  CP_NO_LOAD_BALANCE = 1  /* "flat" sharding of [AG] / [A2A] */
} cp_strategy_t;

typedef enum {
  CP_OK = 0,
  CP_ERR_INVALID_ARG = -1,  /* null pointer, negative size, rank out of range ... */
  CP_ERR_DIVISIBILITY = -2, /* P_i % (2*cp) != 0 (DCS) or T % cp != 0 (NLB) */
  CP_ERR_UNSUPPORTED = -3,  /* head dim other than 64/128, too many heads ... */
  CP_ERR_ALIGNMENT = -4,    /* pointer or row size not 16-byte aligned */
  CP_ERR_CUDA = -5,         /* a CUDA launch or runtime call failed */
  CP_ERR_WORKSPACE = -6,    /* metadata or workspace buffer too small */
  CP_ERR_METADATA = -7,     /* cu_seqlens values inconsistent (device-detected) */
  CP_ERR_TIMEOUT = -8,      /* a bounded device-side wait ran out; results are invalid */
  CP_ERR_RANGE = -9         /* a bf16 value beyond the fp16 range met an fp16 conversion */
} cp_status_t;

/* Type of the attention's tensor-core operands (Q, K, V, dO; the outputs O,
 * dQ and the dK/dV accumulators keep their own types).  With bf16 operands
 * the backward carries P and dS as two bf16 terms (rounded value plus
 * rounding remainder, one extra tensor-core product each) to stay within the
 * 2e-2 bound on long documents; fp16 operands carry 11 significant bits and
 * need one term.  bf16 inputs convert to fp16 exactly when |x| lies in
 * [2^-14, 65504] (cp_thd_gather_f16); smaller values lose low bits (absolute
 * error below 2^-25), larger ones do not fit. */
typedef enum { CP_OPERAND_BF16 = 0, CP_OPERAND_F16 = 1 } cp_dtype_t;

/* Human-readable name of a status code (static storage). */
const char* cp_status_string(int status);

/* ABI version of this header (major*100 + minor). */
int cp_version(void);

/* ---------------------------------------------------------------------------
 * Host-side metadata helpers (host pointers, no GPU work).
 * ------------------------------------------------------------------------- */

/* pad_between_seqs decided from VALUES, never from object identity
 * ([P2P] §Describe the bug, §Expected behavior): *out = 1 when any of the
 * n_docs+1 entries of cu_host and cup_host differ, else 0.  cup_host == NULL
 * means "no padded offsets given" and yields 0.  cu_host, out must be
 * non-NULL; n_docs >= 0. */
int cp_detect_pad_between_seqs(const int32_t* cu_host, const int32_t* cup_host, int n_docs,
                               int* out);

/* Checks host copies of the offsets against the strategy's constraints:
 * cup[0]==0, cup[n]==total_tokens, cup non-decreasing; with pad_between_seqs,
 * cu[0]==0 and 0 <= L_i <= P_i; DCS: P_i % (2*cp_size) == 0; NLB:
 * total_tokens % cp_size == 0.  Returns CP_OK or the first violation. */
int cp_validate_seqlens(const int32_t* cu_host, const int32_t* cup_host, int n_docs,
                        int64_t total_tokens, int cp_size, cp_strategy_t strategy,
                        int pad_between_seqs);

/* Host-known valid end of a layout: one past the last real-token row.
 * rank in [0, cp_size): rank-local layout under `strategy`;
 * rank == -1: the full packed layout.  Used to gate cp_zero_tail. */
int cp_valid_end(const int32_t* cu_host, const int32_t* cup_host, int n_docs, int cp_size,
                 int rank, cp_strategy_t strategy, int pad_between_seqs, int64_t* out);

/* ---------------------------------------------------------------------------
 * Partition index ([AG] §What changed: native THD partition index for CUDA
 * batch slicing; metadata keeps logical document boundaries).
 * ------------------------------------------------------------------------- */

/* Bytes of device metadata cp_partition_index writes for one rank
 * (s_local = total_tokens / cp_size): a 64-byte header, a segment table
 * (32 bytes x (2*n_docs+2)), two int32 tables of s_local entries (each local
 * row's document start and last attended key, -1 for padding rows) and
 * 64-byte block lists, one per 128-row query tile and one per 128-key block.
 * Returns 0 for invalid sizes (total_tokens not divisible by cp_size). */
size_t cp_meta_bytes(int n_docs, int64_t total_tokens, int cp_size);

/* One launch.  Reads d_cu / d_cup (device, int32 [n_docs+1]; d_cu is only
 * read when pad_between_seqs != 0) and writes, for rank `rank`:
 *   d_idx[s_local]     global row of each local row, in local order;
 *   d_restore[...]     (nullable) d_restore[d_idx[t]] = rank*s_local + t, i.e.
 *                      this rank's entries of the inverse of the
 *                      rank-concatenated partition (the K/V restore index of
 *                      [AG] §Sequence Diagram; call once per rank to fill all
 *                      total_tokens entries);
 *   d_meta[meta_bytes] the rank's segment table and per-row tables consumed
 *                      by the attention kernels.
 * s_local = total_tokens / cp_size.  Offsets that break the strategy's
 * constraints set the header status (CP_ERR_DIVISIBILITY / CP_ERR_METADATA)
 * and the device status word; idx/restore are then left unwritten. */
int cp_partition_index(const int32_t* d_cu, const int32_t* d_cup, int n_docs,
                       int64_t total_tokens, int cp_size, int rank, cp_strategy_t strategy,
                       int pad_between_seqs, int32_t* d_idx, int32_t* d_restore, void* d_meta,
                       size_t meta_bytes, void* stream);

/* Every rank's cp_partition_index in ONE launch (one CTA per rank): rank r
 * writes d_idx_all[r*s_local .. (r+1)*s_local) (the ranks' indices side by
 * side, i.e. the index of the rank-concatenated layout), its entries of
 * d_restore (nullable; all total_tokens entries are written) and its
 * metadata at d_meta + r*meta_stride.  meta_stride >= cp_meta_bytes and a
 * multiple of 16 (else CP_ERR_WORKSPACE / CP_ERR_ALIGNMENT).  Results are
 * byte for byte those of the cp_size single-rank calls. */
int cp_partition_index_all(const int32_t* d_cu, const int32_t* d_cup, int n_docs,
                           int64_t total_tokens, int cp_size, cp_strategy_t strategy,
                           int pad_between_seqs, int32_t* d_idx_all, int32_t* d_restore,
                           void* d_meta, size_t meta_stride, void* stream);

/* ---------------------------------------------------------------------------
 * THD row gather / scatter: the index_select restore/unrestore of [AG]
 * §Sequence Diagram, bandwidth bound per [A2A] (paragraph on the 8xH200
 * measurement).  Up to 4 tensors share one index and one launch.
 * ------------------------------------------------------------------------- */

/* d_dst[k] row i = d_src[k] row d_idx[i], i in [0, n_rows), for k < n_tensors.
 * d_src / d_dst are HOST arrays of n_tensors DEVICE pointers; rows are
 * row_bytes long (row_bytes % 16 == 0); d_idx is device int32 [n_rows] with
 * values in [0, src_rows) (a value outside is skipped and sets the device
 * status word).  Destinations must not overlap sources. */
int cp_thd_gather(const void* const* d_src, void* const* d_dst, int n_tensors,
                  const int32_t* d_idx, int64_t n_rows, int64_t src_rows, int64_t row_bytes,
                  void* stream);

/* d_dst[k] row d_idx[i] = d_src[k] row i, i in [0, n_rows).  d_idx values in
 * [0, dst_rows) and pairwise distinct (an injective map; duplicates give an
 * unspecified winner). */
int cp_thd_scatter(const void* const* d_src, void* const* d_dst, int n_tensors,
                   const int32_t* d_idx, int64_t n_rows, int64_t dst_rows, int64_t row_bytes,
                   void* stream);

/* cp_thd_gather that converts bf16 source rows to fp16 (the tensor-core
 * operand type CP_OPERAND_F16): d_dst[k] row i = fp16(d_src[k] row
 * (d_idx ? d_idx[i] : i)), element-wise, round to nearest.  d_idx nullable
 * (identity, src_rows >= n_rows).  A finite value beyond the fp16 range
 * (|x| > 65504) is written as +-65504 and sets the device status word to
 * CP_ERR_RANGE (results computed from it are not valid); infinities and NaN
 * keep their meaning.  Other arguments as cp_thd_gather. */
int cp_thd_gather_f16(const void* const* d_src, void* const* d_dst, int n_tensors,
                      const int32_t* d_idx, int64_t n_rows, int64_t src_rows, int64_t row_bytes,
                      void* stream);

/* Emulated reduce-scatter epilogue of the dK/dV path ([AG] §Sequence Diagram,
 * "unrestore dK/dV for reduce-scatter"): the fp32 accumulators hold the sum
 * over ranks of the per-rank partials in original order; rank r's local
 * gradient is that sum gathered by its partition index and rounded to bf16:
 *   d_dst[k] row t = bf16(d_accum[k] row (d_idx ? d_idx[t] : row0 + t)).
 * Rows are H*D values: fp32 in, bf16 out.  d_accum / d_dst are host arrays of
 * n_tensors (<= 4) device pointers. */
int cp_reduce_scatter_emul(const float* const* d_accum, void* const* d_dst, int n_tensors,
                           const int32_t* d_idx, int64_t row0, int64_t n_rows,
                           int64_t accum_rows, int H, int D, void* stream);

/* Direction of cp_a2a_exchange. */
typedef enum {
  CP_A2A_SEQ_TO_HEAD = 0, /* before attention: token shards -> full sequence, head slice */
  CP_A2A_HEAD_TO_SEQ = 1  /* after attention: full sequence, head slice -> token shards */
} cp_a2a_dir_t;

/* All-to-all exchange of the a2a comm type ("[PyTorch] Extend no-load-balance
 * CP to the a2a comm type", ¶1-2, §Diagram), every rank on one GPU.  The
 * exchange trades token shards for head slices: rank r ends up with all T
 * tokens of heads [r*H/cp, (r+1)*H/cp), which makes its attention a cp_size = 1
 * problem on that slice.
 *   sequence side: [T, H, D] rank-concatenated buffer (rank r's token shard
 *     is rows [r*T/cp, (r+1)*T/cp)).
 *   head side: cp buffers [T, H/cp, D] side by side ([cp, T, H/cp, D]); rank
 *     r's holds every token in original order and heads [r*H/cp, (r+1)*H/cp).
 *   d_perm (device int32 [T], nullable): sequence-side row of original token
 *     g -- the restore index of DUAL_CHUNK_SWAP, which folds the dual-chunk
 *     reorder into the same pass; NULL for flat (NO_LOAD_BALANCE) sharding,
 *     whose rank-concatenated order already is the original order.  It must
 *     be a permutation of [0, T); a value outside is skipped and sets the
 *     device status word.
 * SEQ_TO_HEAD reads d_src[k] (sequence side) and writes d_dst[k] (head side);
 * HEAD_TO_SEQ the reverse.  d_src / d_dst: host arrays of n_tensors (<= 4)
 * device pointers, 16-byte aligned; (H/cp)*D*2 must be a multiple of 16 and H
 * a multiple of cp_size (else CP_ERR_ALIGNMENT / CP_ERR_INVALID_ARG before any
 * launch).  Bit copy.  Destinations must not overlap sources. */
int cp_a2a_exchange(const void* const* d_src, void* const* d_dst, int n_tensors,
                    const int32_t* d_perm, int64_t total_tokens, int cp_size, int H, int D,
                    cp_a2a_dir_t dir, void* stream);

/* Gradient tail-zeroing ([P2P] §Describe the bug, last paragraph; §Expected
 * behavior: gated when no tail exists, graph-safe).  Zeroes rows
 * [valid_end, rows) of each of n_tensors (<= 4) tensors of row_bytes-long rows.
 *   valid_end >= 0: host-known; valid_end == rows launches NOTHING.
 *   valid_end <  0: read *d_valid_end on the device (graph-safe form; one
 *                   launch that exits early when there is no tail).
 * *launched (nullable host int) reports whether a kernel was launched.
 * valid_end = 0 zeroes whole tensors (used to clear dK/dV accumulators). */
int cp_zero_tail(void* const* d_rows, int n_tensors, int64_t rows, int64_t row_bytes,
                 int64_t valid_end, const int32_t* d_valid_end, void* stream, int* launched);

/* ---------------------------------------------------------------------------
 * Causal varlen attention of one rank's local queries against the full K/V
 * ([AG] §Why, §Scope and constraints: causal, window_size=(-1,0), document
 * boundaries from THD metadata).  For local row t at global row g of document
 * i: keys j in [cup[i], g] when g is a real token; padding rows get O = 0,
 * LSE = -inf, dQ = 0.  Scores s = softmax_scale * q.k; LSE in natural log.
 * DUAL_CHUNK_SWAP's two chunks per rank are handled in ONE launch.
 * ------------------------------------------------------------------------- */

/* q_local [s_local,H,D] (rank-local order); k_full, v_full [T,H,D] in
 * original order (the restored all-gather), all three of operand_dtype (bf16
 * or fp16); o_local [s_local,H,D] bf16;
 * lse_local [H, s_local] fp32.  o_resid_local (nullable) [s_local,H,D] bf16
 * receives O's rounding remainder, O - bf16(O), rounded to bf16: O_local +
 * o_resid_local carries the output to about 16 bits, and the backward's
 * Delta = rowsum(dO * O) taken from that sum keeps dQ/dK within the bf16
 * tolerance on long documents (Delta from the bf16 O alone does not).
 * d_meta is the rank's metadata from cp_partition_index (same cp_size, rank,
 * strategy).  D in {64, 128}; H*D*2 <= 65535*16.  Deterministic. */
int cp_attn_fwd(const void* q_local, const void* k_full, const void* v_full, void* o_local,
                void* o_resid_local, float* lse_local, const void* d_meta, size_t meta_bytes,
                int64_t total_tokens, int H, int D, int cp_size, int rank,
                cp_strategy_t strategy, float softmax_scale, cp_dtype_t operand_dtype,
                void* stream);

/* cp_attn_fwd with the partition gather of the queries fused into the kernel
 * (the index_select of get_batch_on_this_cp_rank, [AG] §Sequence Diagram,
 * done by the attention's own loads): query row t of this
 * rank is row d_idx[t] of q_src [src_rows, H, D] of operand_dtype (e.g. the unsharded
 * batch with d_idx from cp_partition_index), so no q_local copy is made.
 * d_idx: device int32 [s_local], 4-byte aligned (a rank's slice of the
 * ranks' indices side by side qualifies); a value outside
 * [0, src_rows) reads row 0 instead and sets the device status word
 * (CP_ERR_INVALID_ARG).  Everything else, including the results, as for
 * cp_attn_fwd: the output is bitwise the same as cp_attn_fwd on the gathered
 * q_local. */
int cp_attn_fwd_gather(const void* q_src, int64_t src_rows, const int32_t* d_idx,
                       const void* k_full, const void* v_full, void* o_local,
                       void* o_resid_local, float* lse_local, const void* d_meta,
                       size_t meta_bytes, int64_t total_tokens, int H, int D, int cp_size,
                       int rank, cp_strategy_t strategy, float softmax_scale,
                       cp_dtype_t operand_dtype, void* stream);

/* Device scratch cp_attn_bwd needs: Delta = rowsum(dO * O), fp32 [H, s_local]. */
size_t cp_attn_bwd_workspace_bytes(int64_t s_local, int H);

/* Backward of cp_attn_fwd for one rank.  Inputs as for cp_attn_fwd plus
 * o_local / lse_local from the forward, o_resid_local (nullable) from the
 * forward's o_resid_local output, and do_local [s_local,H,D] of operand_dtype
 * (like q_local, k_full, v_full).
 * Writes dq_local [s_local,H,D] bf16 (overwritten) and ADDS this rank's
 * partial dK/dV into dk_accum / dv_accum (fp32 [T,H,D], original order; zero
 * them before rank 0 -- e.g. cp_zero_tail with valid_end = 0 -- or start the
 * sum with cp_attn_bwd_ex in CP_BWD_STORE mode).  Each element receives
 * exactly one fp32 addition per call, so calling the ranks in a fixed order
 * on one stream gives a bitwise deterministic sum.  d_workspace:
 * cp_attn_bwd_workspace_bytes bytes of device scratch, contents need not be
 * initialised. */
int cp_attn_bwd(const void* q_local, const void* k_full, const void* v_full, const void* o_local,
                const void* o_resid_local, const float* lse_local, const void* do_local,
                void* dq_local, float* dk_accum,
                float* dv_accum, const void* d_meta, size_t meta_bytes, int64_t total_tokens,
                int H, int D, int cp_size, int rank, cp_strategy_t strategy, float softmax_scale,
                cp_dtype_t operand_dtype, void* d_workspace, size_t workspace_bytes,
                void* stream);

/* How cp_attn_bwd_ex delivers its gradients: one dK/dV choice (bit 0) OR'd
 * with at most one dQ choice (bits 1-2). */
typedef enum {
  CP_BWD_ACCUMULATE = 0,       /* dK/dV: add into the buffers (cp_attn_bwd) */
  CP_BWD_STORE = 1,            /* dK/dV: store into the buffers, every row written */
  CP_BWD_DQ_F32_STORE = 2,     /* dq_local is fp32 [s_local,H,D]: stored, every row */
  CP_BWD_DQ_F32_ACCUMULATE = 4 /* dq_local is fp32 [s_local,H,D]: added into */
} cp_bwd_mode_t;

/* cp_attn_bwd with a choice of mode.  CP_BWD_STORE writes every element of
 * dk_accum / dv_accum (rows that no query of this rank attends get +0.0), so
 * the first rank of the emulated reduce-scatter needs no cleared buffers: the
 * sum started by CP_BWD_STORE on one rank and continued by CP_BWD_ACCUMULATE
 * on the others, in a fixed order on one stream, is bitwise the sum over
 * cleared buffers (a stored partial is p + 0.0, like the first addition).
 * Without a dQ bit dq_local is bf16 and overwritten, as in cp_attn_bwd.  The
 * dQ bits make dq_local an fp32 buffer, for sums of several calls over the
 * same queries (the ring steps of cp_p2p_index): CP_BWD_DQ_F32_STORE starts
 * the sum (every row written, +0.0 where nothing is attended) and
 * CP_BWD_DQ_F32_ACCUMULATE adds one fp32 term per element and call.
 * Same arguments, results and errors as cp_attn_bwd otherwise; an unknown
 * bit, or both dQ bits, returns CP_ERR_INVALID_ARG. */
int cp_attn_bwd_ex(const void* q_local, const void* k_full, const void* v_full,
                   const void* o_local, const void* o_resid_local, const float* lse_local,
                   const void* do_local,
                   void* dq_local, float* dk_accum, float* dv_accum, const void* d_meta,
                   size_t meta_bytes, int64_t total_tokens, int H, int D, int cp_size, int rank,
                   cp_strategy_t strategy, float softmax_scale, cp_dtype_t operand_dtype,
                   cp_bwd_mode_t mode, void* d_workspace, size_t workspace_bytes, void* stream);

/* Scratch cp_attn_bwd_grouped needs: every rank's Delta (fp32 [cp][H][s_local])
 * and the key blocks' work order (12 bytes per 128-key block). */
size_t cp_attn_bwd_grouped_workspace_bytes(int64_t s_local, int H, int cp_size,
                                           int64_t total_tokens);

/* The backward of every rank of an all-gather CP group in one call, with the
 * emulated reduce-scatter's sum done inside the dK/dV kernel ([AG] §Sequence
 * Diagram: per-rank partial dK/dV, summed over the group): each 128-key block
 * walks the attending query tiles of all cp_size ranks and its dK/dV are
 * stored once.  Operands are the ranks' tensors side by side: q_all, o_all,
 * o_resid_all (nullable), do_all and dq_all are [cp_size*s_local, H, D] with
 * rank r's rows at r*s_local (dq_all bf16, overwritten); lse_all is fp32
 * [cp_size][H][s_local]; d_meta_all holds the ranks' metadata meta_stride
 * bytes apart (as cp_partition_index_all writes it; meta_stride % 16 == 0).
 * dk_accum / dv_accum (fp32 [T,H,D], original order) are stored, every
 * element written (+0.0 where no query attends): the sum cp_attn_bwd_ex gives
 * with CP_BWD_STORE on rank 0 and CP_BWD_ACCUMULATE on the others, with the
 * ranks' terms accumulated in the tensor-core products instead of one fp32
 * addition per rank (a different rounding order; deterministic).  dq_all is
 * exactly what cp_attn_bwd gives rank by rank.  Launches: cp_size Delta and
 * cp_size dQ kernels, one ordering kernel and one dK/dV kernel.  Errors as
 * cp_attn_bwd; rank r's metadata must be rank r's (else CP_ERR_METADATA on
 * the device status word and dK/dV are not written). */
int cp_attn_bwd_grouped(const void* q_all, const void* k_full, const void* v_full,
                        const void* o_all, const void* o_resid_all, const float* lse_all,
                        const void* do_all, void* dq_all, float* dk_accum, float* dv_accum,
                        const void* d_meta_all, size_t meta_stride, int64_t total_tokens, int H,
                        int D, int cp_size, cp_strategy_t strategy, float softmax_scale,
                        cp_dtype_t operand_dtype, void* d_workspace, size_t workspace_bytes,
                        void* stream);

/* cp_attn_bwd_grouped with the whole emulated reduce-scatter inside the dK/dV
 * kernel ([AG] §Sequence Diagram: the partial dK/dV are summed over the group
 * and each rank keeps its own rows): the sum over the ranks is taken in the
 * tensor-core products as in cp_attn_bwd_grouped, and the dK/dV kernel's
 * epilogue writes it, rounded to bf16, straight into the rank-concatenated
 * outputs -- the result cp_reduce_scatter_emul gives from cp_attn_bwd_grouped's
 * fp32 sums, bit for bit, without the fp32 buffers and the extra pass.
 *   dk_all / dv_all: bf16 [T, H, D], rank r's rows at r * s_local in its
 *     partition order (overwritten, every row written).
 *   d_restore: device int32 [T], the rank-concatenated row of global row j
 *     (cp_partition_index_all's restore index); required for
 *     DUAL_CHUNK_SWAP, NULL for NO_LOAD_BALANCE (rank-concatenated order is
 *     the original order).  An entry outside [0, T) skips that row and sets
 *     the device status word (CP_ERR_INVALID_ARG).
 * Other arguments, workspace (cp_attn_bwd_grouped_workspace_bytes), launches
 * and errors as cp_attn_bwd_grouped; dk_all / dv_all 16-byte aligned. */
int cp_attn_bwd_grouped_rs(const void* q_all, const void* k_full, const void* v_full,
                           const void* o_all, const void* o_resid_all, const float* lse_all,
                           const void* do_all, void* dq_all, void* dk_all, void* dv_all,
                           const int32_t* d_restore, const void* d_meta_all, size_t meta_stride,
                           int64_t total_tokens, int H, int D, int cp_size,
                           cp_strategy_t strategy, float softmax_scale, cp_dtype_t operand_dtype,
                           void* d_workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * The P2P (ring) comm type, every rank on one GPU ([P2P] §Describe the bug:
 * the P2P context-parallel path, whose per-step sequence metadata comes from
 * repeated get_cu_seqlens_on_cp_rank calls).  At ring step i = 0..cp_size-1
 * rank r holds the K/V shard of rank j = (r - i) mod cp_size (its partition
 * rows, DUAL_CHUNK_SWAP or NO_LOAD_BALANCE) and attends its own queries to
 * it.  Under both strategies every query row sees one contiguous run of the
 * shard's rows, so a step is a cp_size = 1 attention call:
 *   cp_attn_fwd(q_local, k_shard_j, v_shard_j, o_i, lse_i, step meta,
 *               total_tokens = s_local, cp_size = 1, rank = 0, strategy, ...)
 * the steps' partial outputs are combined by cp_p2p_merge, and the backward
 * runs per step with the merged O / LSE (dQ summed over the steps in fp32,
 * dK/dV of shard j summed over the ranks that attended it).
 * ------------------------------------------------------------------------- */

/* Bytes of ONE ring step's metadata (a multiple of 16); a rank's metadata is
 * cp_size of these blocks back to back, step i at i * cp_p2p_meta_bytes.
 * Returns 0 for invalid sizes (total_tokens not divisible by cp_size). */
size_t cp_p2p_meta_bytes(int n_docs, int64_t total_tokens, int cp_size);

/* One launch (one CTA per step): the metadata of all cp_size ring steps of
 * rank `rank`.  Step i's block describes queries = this rank's s_local local
 * rows, keys = the s_local local rows of rank (rank - i) mod cp_size, with
 * header cp_size = 1, rank = 0, total_tokens = s_local and the given strategy
 * (the values the step's attention call passes); its row tables hold each
 * query row's first and last visible key row of the shard (0 / -1 when it sees
 * none: padding rows, and rows whose document has no earlier key in that
 * shard).  d_cu / d_cup / pad_between_seqs as for cp_partition_index.
 * d_meta: >= cp_size * cp_p2p_meta_bytes bytes, 16-byte aligned.  Offsets
 * that break the strategy's constraints set every step's header status and
 * the device status word. */
int cp_p2p_index(const int32_t* d_cu, const int32_t* d_cup, int n_docs, int64_t total_tokens,
                 int cp_size, int rank, cp_strategy_t strategy, int pad_between_seqs,
                 void* d_meta, size_t meta_bytes, void* stream);

/* Combination of n_steps partial attention outputs of the same queries over
 * disjoint key sets (the ring steps): with l_i = lse_steps[i],
 *   lse = log(sum_i exp(l_i)),   out = sum_i exp(l_i - lse) * o_i,
 * in fp32, out rounded to bf16 once; rows with every l_i = -inf get lse = -inf
 * and out = 0.  d_o_steps: bf16 [n_steps, s_local, H, D]; d_lse_steps: fp32
 * [n_steps, H, s_local] (natural log, as cp_attn_fwd writes it); d_out: bf16
 * [s_local, H, D]; d_lse: fp32 [H, s_local].  d_o_steps_resid (nullable, same
 * layout as d_o_steps): the steps' O rounding remainders (cp_attn_fwd's
 * o_resid_local output), added to o_i before weighting; d_out_resid
 * (nullable, like d_out): receives the merged output's own bf16 rounding
 * remainder, for the backward's Delta.  D in {64, 128}.  One launch. */
int cp_p2p_merge(const void* d_o_steps, const void* d_o_steps_resid, const float* d_lse_steps,
                 int n_steps, int64_t s_local, int H, int D, void* d_out, void* d_out_resid,
                 float* d_lse, void* stream);

/* Scratch cp_attn_bwd_ring needs: every rank's Delta (fp32 [cp][H][s_local])
 * and the work orders (12 bytes per 128-key block of every shard). */
size_t cp_attn_bwd_ring_workspace_bytes(int64_t s_local, int H, int cp_size);

/* The backward of every rank of the P2P ring in one pass per gradient: the
 * result of the per-step backward (cp_attn_bwd_ex at every ring step with the
 * merged O / LSE, dQ summed over a rank's steps, dK/dV of shard j summed over
 * the ranks that attended it), with every sum formed inside the kernels.  Per
 * rank one dQ launch walks the rank's ring steps in ring order (dq_all, bf16,
 * stored once); one dK/dV launch covers the 128-key blocks of every shard,
 * each walking the query tiles of the ranks that hold that shard at some step,
 * and stores dk_accum / dv_accum once (fp32 [cp_size*s_local, H, D],
 * rank-concatenated rows, +0.0 where nothing attends).  Operands are the
 * ranks' tensors side by side: q_all, o_all, o_resid_all (nullable), do_all,
 * dq_all [cp_size*s_local, H, D]; k_shards / v_shards the ranks' K/V shards
 * side by side; lse_all fp32 [cp_size][H][s_local].  d_ring_meta: rank r's
 * step metadata at r*rank_stride, step i at +i*step_bytes (cp_p2p_index
 * output; rank_stride >= cp_size*step_bytes, both % 16 == 0).  s_local must be
 * a multiple of 32 (else CP_ERR_UNSUPPORTED: a shard's output chunks would
 * reach into the next shard).  Launches: cp_size Delta, per rank an ordering
 * kernel and a dQ kernel, one ordering kernel and one dK/dV kernel.
 * Deterministic.  Errors as cp_attn_bwd; every step header is checked on the
 * device (CP_ERR_METADATA, gradients not written). */
int cp_attn_bwd_ring(const void* q_all, const void* k_shards, const void* v_shards,
                     const void* o_all, const void* o_resid_all, const float* lse_all,
                     const void* do_all, void* dq_all, float* dk_accum, float* dv_accum,
                     const void* d_ring_meta, size_t step_bytes, size_t rank_stride,
                     int64_t s_local, int H, int D, int cp_size, cp_strategy_t strategy,
                     float softmax_scale, cp_dtype_t operand_dtype, void* d_workspace,
                     size_t workspace_bytes, void* stream);

/* cp_attn_bwd_ring with the reduce-scatter's cast in the dK/dV kernel's
 * epilogue: dk_all / dv_all are bf16 [cp_size*s_local, H, D] (rank-concatenated
 * shards, the ring's own layout, so no index is needed), every row written, each
 * value the bf16 rounding of the fp32 sum cp_attn_bwd_ring stores (bitwise what
 * cp_reduce_scatter_emul makes of it).  Other arguments, workspace
 * (cp_attn_bwd_ring_workspace_bytes), launches and errors as cp_attn_bwd_ring;
 * dk_all / dv_all 16-byte aligned. */
int cp_attn_bwd_ring_rs(const void* q_all, const void* k_shards, const void* v_shards,
                        const void* o_all, const void* o_resid_all, const float* lse_all,
                        const void* do_all, void* dq_all, void* dk_all, void* dv_all,
                        const void* d_ring_meta, size_t step_bytes, size_t rank_stride,
                        int64_t s_local, int H, int D, int cp_size, cp_strategy_t strategy,
                        float softmax_scale, cp_dtype_t operand_dtype, void* d_workspace,
                        size_t workspace_bytes, void* stream);

/* Scratch cp_attn_fwd_ring needs: its work order, 12 bytes per 128-row query
 * tile (16-aligned halves). */
size_t cp_attn_fwd_ring_workspace_bytes(int64_t s_local);

/* Every ring step of rank `rank` in one pass: the result of cp_attn_fwd on
 * each of the n_steps steps followed by cp_p2p_merge, without the partial
 * outputs.  Step i attends q_local to the K/V shard of rank
 * j = (rank - i) mod cp_size, rows [j*s_local, (j+1)*s_local) of k_shards /
 * v_shards ([cp_size*s_local, H, D] of operand_dtype, the ranks' shards side by
 * side); the kernel walks the steps' key blocks in ring order within one
 * online softmax per row, whose rescaling is the merge.  d_step_meta: the
 * rank's step metadata, step_bytes apart, as cp_p2p_index writes it
 * (step_bytes = cp_p2p_meta_bytes, % 16 == 0); n_steps in [1, cp_size] (the
 * ring's steps of the rank: every step for DUAL_CHUNK_SWAP, steps 0..rank for
 * NO_LOAD_BALANCE).  Outputs as cp_attn_fwd: o_local [s_local,H,D] bf16,
 * o_resid_local (nullable) its rounding remainder, lse_local fp32 [H,s_local].
 * The result equals the per-step path up to the rounding order (one fp32
 * online softmax instead of bf16 partials combined in fp32).  Launches: one
 * ordering kernel (the rank's query tiles heaviest first by their block count
 * over the steps) and one attention kernel.  Errors as cp_attn_fwd; every
 * step's header is checked on the device (CP_ERR_METADATA, nothing written). */
int cp_attn_fwd_ring(const void* q_local, const void* k_shards, const void* v_shards,
                     void* o_local, void* o_resid_local, float* lse_local,
                     const void* d_step_meta, size_t step_bytes, int n_steps, int64_t s_local,
                     int H, int D, int cp_size, int rank, cp_strategy_t strategy,
                     float softmax_scale, cp_dtype_t operand_dtype, void* d_workspace,
                     size_t workspace_bytes, void* stream);

/* Largest Delta scratch cp_attn_bwd_noalloc can use: s_local*H <= this many
 * floats (4 MiB of device memory per GPU that loads the library). */
#define CP_NOALLOC_MAX_SCRATCH_FLOATS 1048576

/* cp_attn_bwd without a caller-provided workspace, for callers that cannot
 * allocate device memory at this point of their program: runtimes that hand
 * out device memory only from an arena planned ahead of time, plugins whose
 * host framework owns the device allocator and forbids allocations behind its
 * back, and host code that must not pay the implicit device synchronisation
 * of cudaMalloc/cudaFree.  The pages have no counterpart to this entry point;
 * it only changes where the backward's scratch lives.
 * Same arguments, results and errors as cp_attn_bwd, minus the workspace.
 * The Delta scratch (fp32 [H, s_local]) lives in a fixed device array compiled
 * into the library (CP_NOALLOC_MAX_SCRATCH_FLOATS floats, held on every GPU
 * that loads the library until the process exits); nothing is allocated or
 * freed.  s_local*H above that maximum returns CP_ERR_WORKSPACE before any
 * launch.  The first call on a device looks up that array's device address
 * (with that device current) and keeps it for the device's current context;
 * make that first call before any stream capture.  After a cudaDeviceReset
 * the device gets a new context with the library's module loaded anew, and
 * the first call in it looks the address up again (again: before any
 * capture).  Every call shares the one array and leaves its last
 * contents there; each call rewrites all the scratch it reads before reading
 * it, so nothing has to start at zero.  Calls whose work overlaps on the GPU
 * (other streams, other host threads) race on the array: serialise them. */
int cp_attn_bwd_noalloc(const void* q_local, const void* k_full, const void* v_full,
                        const void* o_local, const void* o_resid_local,
                        const float* lse_local, const void* do_local,
                        void* dq_local, float* dk_accum, float* dv_accum, const void* d_meta,
                        size_t meta_bytes, int64_t total_tokens, int H, int D, int cp_size,
                        int rank, cp_strategy_t strategy, float softmax_scale,
                        cp_dtype_t operand_dtype, void* stream);

/* ---------------------------------------------------------------------------
 * Diagnostics
 * ------------------------------------------------------------------------- */

/* Reads (and when reset != 0 clears) the current device's status word:
 * CP_OK or the first device-detected error since the last reset.  This is
 * the one entry point that synchronises (it waits for all prior work). */
int cp_device_status(int* status, int reset);

#ifdef __cplusplus
}
#endif

#endif /* CPTHD_H */
