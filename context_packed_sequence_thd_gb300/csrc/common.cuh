// common.cuh -- shared host/device definitions of libcpthd (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "cpthd.h"

namespace cpthd {

// ---------------------------------------------------------------------------
// Rank metadata written by the partition kernel and read by the attention
// kernels.  Layout in device memory:
//   [0, 64)                   MetaHeader
//   [64, 64 + 32*max_segs)    Segment[max_segs], sorted by local_start
//   rows_offset:              int32 row_lo[s_local], int32 row_hi[s_local]
//   lists_offset (16-aligned): one 64-byte block list per 128-row query tile
//                             (the key blocks it attends), then one per
//                             128-key block (the query tiles attending it)
//   after the lists:          the work order, int2 {tile, blocks} per tile,
//                             heaviest first: query tiles, then key blocks
// A segment is a maximal run of local rows that are consecutive global rows
// of one document: one DUAL_CHUNK_SWAP chunk, or one document's piece of a
// NO_LOAD_BALANCE range.  Row t of a segment (u = t - local_start) is global
// row global_start + u; it is a real token when u < valid_len.
// row_lo/row_hi: the keys local row t attends are [row_lo[t], row_hi[t]]
// (row_hi = -1, row_lo = 0 for padding rows).
// A block list is int2[8]: {count, blocks} then up to 7 merged, increasing
// inclusive intervals [first, last] of 128-wide block indices; `blocks` is the
// number of blocks the intervals cover.  Entry q of a family's work order is
// {tile, blocks} of the tile with the q-th most blocks (ties by index): the
// attention kernels take their work items heaviest first, and one 8-byte load
// tells a warp which tile comes next and how many blocks it has.
// ---------------------------------------------------------------------------
constexpr int32_t kMetaMagic = 0x43505448;  // "CPTH"
constexpr int kTile = 128;       // query-tile rows and key-block width of the lists
constexpr int kListCap = 7;      // intervals per list (over capacity the last widens)
constexpr int kListBytes = 64;

struct MetaHeader {
  int32_t magic;
  int32_t status;
  int32_t strategy;
  int32_t cp_size;
  int32_t rank;
  int32_t n_docs;
  int32_t s_local;
  int32_t n_segs;
  int32_t valid_end;  // one past the last real-token local row
  int32_t pad_between_seqs;
  int32_t total_tokens;
  int32_t max_segs;
  int32_t seg_offset;    // bytes
  int32_t rows_offset;   // bytes; row_lo at rows_offset, row_hi 4*s_local later
  int32_t lists_offset;  // bytes; query-tile lists, then key-block lists
  int32_t n_kblocks;     // number of 128-key blocks (ceil(total_tokens / 128))
};
static_assert(sizeof(MetaHeader) == 64, "header is 64 bytes");

struct Segment {
  int32_t local_start;
  int32_t global_start;
  int32_t len;
  int32_t doc_lo;     // first row of the document (cup[i])
  int32_t valid_len;  // real-token rows at the start of this segment
  int32_t doc;
  int32_t reserved[2];
};
static_assert(sizeof(Segment) == 32, "segment is 32 bytes");

inline __host__ __device__ int max_segs_for(int n_docs) { return 2 * n_docs + 2; }
inline __host__ __device__ size_t seg_offset_bytes() { return 64; }
inline __host__ __device__ size_t rows_offset_bytes(int n_docs) {
  return 64 + 32 * (size_t)max_segs_for(n_docs);
}
inline __host__ __device__ size_t lists_offset_bytes(int n_docs, int64_t s_local) {
  return (rows_offset_bytes(n_docs) + 8 * (size_t)s_local + 15) & ~(size_t)15;
}
inline __host__ __device__ int64_t n_tiles_of(int64_t rows) { return (rows + kTile - 1) / kTile; }
inline __host__ __device__ size_t meta_bytes_for(int n_docs, int64_t s_local, int cp) {
  const size_t n = (size_t)(n_tiles_of(s_local) + n_tiles_of(s_local * cp));
  return lists_offset_bytes(n_docs, s_local) + (size_t)(kListBytes + 8) * n;
}

// Work item of the j-th round of CTA c among G persistent CTAs: rounds of G
// consecutive items (sorted heaviest first) alternate direction, so every
// CTA's sum of item sizes stays close to the mean.
__host__ __device__ __forceinline__ int snake_item(int j, int c, int G) {
  return j * G + ((j & 1) ? G - 1 - c : c);
}

// Tile rank q (into a heaviest-first order of n_tiles tiles) and head h of
// work item k of a launch over n_tiles * H items, heads taken in groups of G:
// within a group the items are heaviest first across its heads (tile-major),
// groups one after another.  G = H is the globally heaviest-first order (the
// best balance); G = 1 keeps the CTAs on one head at a time, so that head's
// streamed operands stay resident in L2.
__host__ __device__ __forceinline__ void item_of(int k, int n_tiles, int H, int G, int* q,
                                                 int* h) {
  G = max(1, min(G, H));
  const int group = k / (G * n_tiles);
  const int hg = min(G, H - group * G);  // heads in this group (the last may have fewer)
  const int within = k - group * G * n_tiles;
  *q = within / hg;
  *h = group * G + within % hg;
}

struct MetaView {
  const MetaHeader* hdr;
  const Segment* segs;
  const int32_t* row_lo;
  const int32_t* row_hi;
  const int2* qlists;  // per 128-row query tile: key blocks attended
  const int2* klists;  // per 128-key block: query tiles attending it
  const int2* qorder;  // {tile, blocks} of the query tiles, heaviest first
  const int2* korder;  // {block, tiles} of the key blocks, heaviest first
};

inline __device__ MetaView meta_view(const void* meta) {
  MetaView v;
  const char* base = reinterpret_cast<const char*>(meta);
  v.hdr = reinterpret_cast<const MetaHeader*>(base);
  v.segs = reinterpret_cast<const Segment*>(base + v.hdr->seg_offset);
  v.row_lo = reinterpret_cast<const int32_t*>(base + v.hdr->rows_offset);
  v.row_hi = v.row_lo + v.hdr->s_local;
  v.qlists = reinterpret_cast<const int2*>(base + v.hdr->lists_offset);
  v.klists = v.qlists + (kListBytes / 8) * n_tiles_of(v.hdr->s_local);
  v.qorder = v.klists + (kListBytes / 8) * v.hdr->n_kblocks;
  v.korder = v.qorder + n_tiles_of(v.hdr->s_local);
  return v;
}

// The metadata header belongs to this call and its tables lie inside the
// caller's buffer of meta_bytes.
inline __device__ bool meta_matches(const MetaHeader* h, size_t meta_bytes, int T, int s_local,
                                    int cp, int rank, int strategy) {
  const int64_t lists_end = (int64_t)h->lists_offset + (int64_t)(kListBytes + 8) *
                                                         (n_tiles_of(s_local) + (int64_t)h->n_kblocks);
  const bool fits = h->n_segs >= 0 && h->n_segs <= h->max_segs && h->seg_offset == 64 &&
                    (int64_t)h->rows_offset >= 64 + 32 * (int64_t)h->max_segs &&
                    (int64_t)h->lists_offset >= (int64_t)h->rows_offset + 8 * (int64_t)s_local &&
                    (h->lists_offset & 15) == 0 && h->n_kblocks == n_tiles_of(T) &&
                    lists_end <= (int64_t)meta_bytes;
  return fits && h->magic == kMetaMagic && h->status == 0 && h->s_local == s_local &&
         h->rank == rank && h->cp_size == cp && h->strategy == strategy && h->total_tokens == T;
}

// Index of the last segment whose local_start <= t (segments are sorted and
// tile [0, s_local) without gaps).
inline __device__ int find_segment_local(const Segment* segs, int n_segs, int t) {
  int lo = 0, hi = n_segs - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (segs[mid].local_start <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Index of the first segment whose global range ends after key j, i.e.
// global_start + len > j (global ranges increase with the segment index).
inline __device__ int find_segment_global_end(const Segment* segs, int n_segs, int j) {
  int lo = 0, hi = n_segs;
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if (segs[mid].global_start + segs[mid].len > j) hi = mid; else lo = mid + 1;
  }
  return lo;
}

// Key-block intervals [first, last] (inclusive, block size BN) that the local
// query rows [t0, t0+rows) attend, merged and in increasing order.  Written to
// out[] (capacity cap); returns the number of intervals.  One thread.
inline __device__ int build_kv_intervals(const MetaView& m, int t0, int rows, int BN, int2* out,
                                         int cap) {
  const int n_segs = m.hdr->n_segs;
  if (n_segs <= 0) return 0;
  int k = find_segment_local(m.segs, n_segs, t0);
  int next = 0, count = 0;
  const int t1 = t0 + rows;
  for (; k < n_segs; ++k) {
    const Segment s = m.segs[k];
    if (s.local_start >= t1) break;
    int u0 = max(0, t0 - s.local_start);
    int u1 = min(s.valid_len, t1 - s.local_start);
    if (u0 >= u1) continue;
    int first = s.doc_lo / BN;
    int last = (s.global_start + u1 - 1) / BN;
    first = max(first, next);
    if (first > last) continue;
    if (count > 0 && out[count - 1].y + 1 == first) {
      out[count - 1].y = last;
    } else if (count < cap) {
      out[count++] = make_int2(first, last);
    } else {
      out[count - 1].y = last;  // over capacity: widen the last interval (still correct)
    }
    next = last + 1;
  }
  return count;
}

// Query-tile intervals (tiles of BM local rows) whose queries attend at least
// one key in [j0, j1], merged and increasing.  One thread.
inline __device__ int build_q_intervals(const MetaView& m, int j0, int j1, int BM, int2* out,
                                        int cap) {
  const int n_segs = m.hdr->n_segs;
  if (n_segs <= 0) return 0;
  int k = find_segment_global_end(m.segs, n_segs, j0);
  int next = 0, count = 0;
  for (; k < n_segs; ++k) {
    const Segment s = m.segs[k];
    if (s.doc_lo > j1) break;
    // queries of this segment attending some key in [j0, j1]: real tokens at
    // global rows >= max(j0, doc_lo)
    int g_first = max(j0, s.doc_lo);
    int u0 = max(0, g_first - s.global_start);
    int u1 = s.valid_len;
    if (u0 >= u1) continue;
    int first = (s.local_start + u0) / BM;
    int last = (s.local_start + u1 - 1) / BM;
    first = max(first, next);
    if (first > last) continue;
    if (count > 0 && out[count - 1].y + 1 == first) {
      out[count - 1].y = last;
    } else if (count < cap) {
      out[count++] = make_int2(first, last);
    } else {
      out[count - 1].y = last;
    }
    next = last + 1;
  }
  return count;
}

// ---------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------
inline __device__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

inline __device__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (low 16 bits)
  return *reinterpret_cast<uint32_t*>(&v);
}

inline __device__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);  // .x = lo (low 16 bits)
  return *reinterpret_cast<uint32_t*>(&v);
}
// Packs a pair in the tensor-core operand type (fp16 or bf16).
template <bool F16>
inline __device__ uint32_t pack_op(float lo, float hi) {
  return F16 ? pack_f16(lo, hi) : pack_bf16(lo, hi);
}

// The two bf16 values of a packed pair as fp32 (exact: a bf16 is the upper
// half of an fp32 bit pattern).
inline __device__ float bf16_lo_f(uint32_t p) { return __uint_as_float(p << 16); }
inline __device__ float bf16_hi_f(uint32_t p) { return __uint_as_float(p & 0xFFFF0000u); }

}  // namespace cpthd

// host-side helpers shared by the translation units
namespace cpthd_host {
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }
inline int launch_status() {
  return cudaGetLastError() == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}
// SMs of the current device (queried once per translation unit; 148 if the
// query fails, which only sizes grids)
inline int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
      n = v;
    else
      return 148;
  }
  return n;
}
}  // namespace cpthd_host

// per-translation-unit device status word accessors (defined in each .cu)
extern "C" int cpthd_status_partition(int reset);
extern "C" int cpthd_status_rows(int reset);
extern "C" int cpthd_status_attn(int reset);
extern "C" int cpthd_status_fwd_tc(int reset);
extern "C" int cpthd_status_bwd_tc(int reset);

// tcgen05 forward (attn_fwd_tc.cu); arguments validated by cp_attn_fwd /
// cp_attn_fwd_gather (q_idx null: q is the rank's [s_local, H, D] queries;
// o_resid nullable: O's bf16 rounding remainder, as bf16; f16: Q/K/V are fp16,
// else bf16).
// limit_ns bounds every wait (0: the 4 s default); skip_first_k != 0 only in
// the failure-detection test (CTA 0 never loads its first K tile).
int cpthd_attn_fwd_tc(const void* q, const int32_t* q_idx, int q_rows, const void* k,
                      const void* v, void* o, void* o_resid, float* lse, const void* meta,
                      size_t meta_bytes,
                      int T, int H, int D, int s_local, int cp, int rank, int strategy,
                      float scale_log2, int f16, cudaStream_t s, uint64_t limit_ns = 0,
                      int skip_first_k = 0);

// The ring forward in one pass (attn_fwd_tc.cu): every ring step of a rank,
// one online softmax over the steps' shards; scratch: ring_scratch_bytes.
inline __host__ __device__ size_t ring_order_offset(int64_t s_local) {
  return ((size_t)cpthd::n_tiles_of(s_local) * 4 + 15) & ~(size_t)15;
}
inline __host__ __device__ size_t ring_scratch_bytes(int64_t s_local) {
  return ring_order_offset(s_local) + (size_t)cpthd::n_tiles_of(s_local) * 8;
}
int cpthd_attn_fwd_ring_tc(const void* q, const void* k_shards, const void* v_shards, void* o,
                           void* o_resid, float* lse, const void* step_meta, size_t step_bytes,
                           int n_steps, int H, int D, int s_local, int cp, int rank, int strategy,
                           float scale_log2, int f16, void* scratch, cudaStream_t s);

// The ring backward in one pass (attn_bwd_tc.cu); scratch: the work orders
// (the larger of a rank's query tiles and every shard's key blocks).
inline __host__ __device__ size_t ring_bwd_order_offset(int64_t s_local, int cp) {
  return ((size_t)cpthd::n_tiles_of(s_local) * cp * 4 + 15) & ~(size_t)15;
}
inline __host__ __device__ size_t ring_bwd_scratch_bytes(int64_t s_local, int cp) {
  return ring_bwd_order_offset(s_local, cp) + (size_t)cpthd::n_tiles_of(s_local) * cp * 8;
}
int cpthd_attn_bwd_ring_tc(const void* q_all, const void* k_shards, const void* v_shards,
                           const void* dout_all, const float* lse_all, const float* delta_all,
                           void* dq_all, float* dk, float* dv, const void* ring_meta,
                           size_t step_bytes, size_t rank_stride, int H, int D, int s_local,
                           int cp, int strategy, float scale, float scale_log2, int f16,
                           void* scratch, cudaStream_t s, void* dk16 = nullptr,
                           void* dv16 = nullptr);

// tcgen05 dQ and dK/dV kernels (attn_bwd_tc.cu); Delta already in `delta`;
// mode holds cp_bwd_mode_t bits (1: dK/dV stored; 2 / 4: dQ fp32 stored / added)
// and, internally, kBwdDqOnly (the dQ kernel alone); f16: Q/K/V/dO are fp16,
// else bf16
constexpr int kBwdDqOnly = 8;
int cpthd_attn_bwd_tc(const void* q, const void* k, const void* v, const void* dout,
                      const float* lse, const float* delta, void* dq, float* dk, float* dv,
                      const void* meta, size_t meta_bytes, int T, int H, int D, int s_local,
                      int cp, int rank, int strategy, float scale, float scale_log2,
                      int mode, int f16, cudaStream_t s, int pdl = 0);

// Scratch of the rank-grouped dK/dV: n_kb int totals, then (16-aligned) the
// n_kb int2 work order.
inline __host__ __device__ size_t grouped_order_offset(int64_t T) {
  return ((size_t)cpthd::n_tiles_of(T) * 4 + 15) & ~(size_t)15;
}
inline __host__ __device__ size_t grouped_scratch_bytes(int64_t T) {
  return grouped_order_offset(T) + (size_t)cpthd::n_tiles_of(T) * 8;
}

// Rank-grouped dK/dV (attn_bwd_tc.cu): every key block walks the query tiles of
// all cp ranks and is stored once; operands as the per-rank call, concatenated
// over the ranks (see the definition).
int cpthd_attn_dkdv_grouped_tc(const void* q_all, const void* k, const void* v,
                               const void* dout_all, const float* lse_all,
                               const float* delta_all, float* dk, float* dv,
                               const void* meta_all, size_t meta_stride, int T, int H, int D,
                               int s_local, int cp, int strategy, float scale, float scale_log2,
                               int f16, void* scratch, cudaStream_t s,
                               void* dk16 = nullptr, void* dv16 = nullptr,
                               const int32_t* rs_row = nullptr, int pdl = 0);
