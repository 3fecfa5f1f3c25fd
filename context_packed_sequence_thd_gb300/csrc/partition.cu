// partition.cu -- per-rank THD partition index (one launch).
//
// "[PyTorch] Add no-load-balance THD all-gather CP", §What changed / §Why:
// DUAL_CHUNK_SWAP gives rank r chunks r and 2*cp-1-r of every document's
// padded range (2*cp equal chunks); NO_LOAD_BALANCE gives rank r the
// contiguous physical rows [r*s_local, (r+1)*s_local) while the THD metadata
// keeps the logical document boundaries.  The per-rank valid-token counts
// (the quantity the P2P issue's get_cu_seqlens_on_cp_rank helper recomputes
// with many small launches) fall out of the same pass, and so do the block
// lists the attention kernels iterate: for every 128-row query tile the key
// blocks it attends, for every 128-key block the query tiles attending it.
//
// One CTA of 1024 threads per rank (cp_partition_index: one rank;
// cp_partition_index_all: every rank of a plan in one launch): documents are
// processed 1024 at a time; a block-wide exclusive scan (warp __shfl_up_sync
// scans + one scan of the warp totals) turns per-document segment counts and
// local row counts into offsets.  A second pass writes the row tables, one
// warp per segment.
//
// Also the per-step metadata of the P2P ring comm type (p2p_index_kernel,
// one CTA per ring step, every step of a rank in one launch).
#include "common.cuh"

namespace cpthd {

static __device__ int g_status_partition;

namespace {

constexpr int kThreads = 1024;
constexpr int kNbCap = 4096;  // block counts kept in shared memory (16 KB)

// Block-wide exclusive scan of v; *total receives the block sum.  All threads
// of the block must call it.
__device__ int block_exclusive_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < kThreads / 32) ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;  // inclusive prefix of warp totals
  }
  __syncthreads();
  int excl = x - v + (warp > 0 ? s_warp[warp - 1] : 0);
  *total = s_warp[kThreads / 32 - 1];
  __syncthreads();  // s_warp is reused by the next call
  return excl;
}

__device__ __forceinline__ int clampi(int x, int lo, int hi) { return min(max(x, lo), hi); }

// Heaviest-first work order of both list families, {tile, blocks} (a rank by
// comparison against every other tile of the family; stable for equal
// counts).  Counts come from s_nb (when counts_in_smem, indexed like the
// lists), or, for very long sequences, are staged there from the lists in
// chunks.  All threads of the block call it.
__device__ void build_work_order(int2* lists, int n_qt, int n_kb, int* s_nb, bool counts_in_smem) {
  int2* order = lists + (kListBytes / 8) * (n_qt + n_kb);
  for (int fam = 0; fam < 2; ++fam) {
    const int n = fam == 0 ? n_qt : n_kb;
    const int base = fam == 0 ? 0 : n_qt;
    int2* ord = order + base;
    for (int q0 = 0; q0 < n; q0 += kThreads) {
      const int q = q0 + threadIdx.x;
      const int mine = q < n ? lists[(kListBytes / 8) * (base + q)].y : 0;
      int rank = 0;
      if (counts_in_smem) {
        if (q < n)
          for (int i = 0; i < n; ++i) {
            const int o = s_nb[base + i];
            rank += (o > mine || (o == mine && i < q)) ? 1 : 0;
          }
      } else {
        for (int c0 = 0; c0 < n; c0 += kNbCap) {
          const int cn = min(kNbCap, n - c0);
          __syncthreads();
          for (int i = threadIdx.x; i < cn; i += kThreads)
            s_nb[i] = lists[(kListBytes / 8) * (base + c0 + i)].y;
          __syncthreads();
          if (q < n)
            for (int i = 0; i < cn; ++i) {
              const int o = s_nb[i];
              rank += (o > mine || (o == mine && c0 + i < q)) ? 1 : 0;
            }
        }
      }
      if (q < n) ord[rank] = make_int2(q, mine);
    }
  }
}


__global__ void __launch_bounds__(kThreads, 1)
partition_kernel(const int32_t* __restrict__ cu, const int32_t* __restrict__ cup, int n_docs,
                 int T, int cp, int rank0, int strategy, int pad, int32_t* __restrict__ idx0,
                 int32_t* __restrict__ restore, char* __restrict__ meta0, size_t meta_stride) {
  // CTA b builds rank rank0 + b: its index at idx0 + b*s_local, its metadata
  // at meta0 + b*meta_stride (one CTA per rank, ranks independent)
  const int rank = rank0 + blockIdx.x;
  int32_t* idx = idx0 + (size_t)blockIdx.x * (T / cp);
  char* meta = meta0 + (size_t)blockIdx.x * meta_stride;
  __shared__ int s_warp[32];
  __shared__ int s_err;
  __shared__ int s_valid_end;
  __shared__ int s_carry_segs, s_carry_rows;
  __shared__ int s_nb[kNbCap];

  MetaHeader* hdr = reinterpret_cast<MetaHeader*>(meta);
  Segment* segs = reinterpret_cast<Segment*>(meta + seg_offset_bytes());
  const int s_local = T / cp;
  const int max_segs = max_segs_for(n_docs);
  int32_t* row_lo = reinterpret_cast<int32_t*>(meta + rows_offset_bytes(n_docs));
  int32_t* row_hi = row_lo + s_local;
  const int R0 = rank * s_local, R1 = R0 + s_local;

  if (threadIdx.x == 0) {
    int e = 0;
    if (cup[0] != 0 || cup[n_docs] != T) e = CP_ERR_METADATA;
    if (pad && cu[0] != 0) e = CP_ERR_METADATA;
    s_err = e;
    s_valid_end = 0;
    s_carry_segs = 0;
    s_carry_rows = 0;
  }
  __syncthreads();

  for (int base = 0; base < n_docs; base += kThreads) {
    const int i = base + threadIdx.x;
    int nseg = 0, nrows = 0, a = 0, P = 0, L = 0, c = 0, lo = 0, hi = 0;
    if (i < n_docs) {
      a = cup[i];
      P = cup[i + 1] - a;
      L = pad ? (cu[i + 1] - cu[i]) : P;
      if (P < 0 || L < 0 || L > P) atomicCAS(&s_err, 0, CP_ERR_METADATA);
      if (strategy == CP_DUAL_CHUNK_SWAP) {
        if (P > 0 && (P % (2 * cp)) != 0) atomicCAS(&s_err, 0, CP_ERR_DIVISIBILITY);
        c = P / (2 * cp);
        nseg = (c > 0) ? 2 : 0;
        nrows = 2 * c;
      } else {
        lo = max(a, R0);
        hi = min(a + max(P, 0), R1);
        nrows = max(0, hi - lo);
        nseg = nrows > 0 ? 1 : 0;
      }
    }
    int tot_segs, tot_rows;
    const int seg_off = block_exclusive_scan(nseg, s_warp, &tot_segs) + s_carry_segs;
    const int row_off = block_exclusive_scan(nrows, s_warp, &tot_rows) + s_carry_rows;
    if (i < n_docs && nseg > 0 && seg_off + nseg <= max_segs) {
      if (strategy == CP_DUAL_CHUNK_SWAP) {
        const int chunks[2] = {rank, 2 * cp - 1 - rank};
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          Segment s;
          s.local_start = row_off + q * c;
          s.global_start = a + chunks[q] * c;
          s.len = c;
          s.doc_lo = a;
          s.valid_len = clampi(L - chunks[q] * c, 0, c);
          s.doc = i;
          s.reserved[0] = s.reserved[1] = 0;
          segs[seg_off + q] = s;
          if (s.valid_len > 0) atomicMax(&s_valid_end, s.local_start + s.valid_len);
        }
      } else {
        Segment s;
        s.local_start = lo - R0;
        s.global_start = lo;
        s.len = nrows;
        s.doc_lo = a;
        s.valid_len = clampi(a + L - lo, 0, nrows);
        s.doc = i;
        s.reserved[0] = s.reserved[1] = 0;
        segs[seg_off] = s;
        if (s.valid_len > 0) atomicMax(&s_valid_end, s.local_start + s.valid_len);
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      s_carry_segs += tot_segs;
      s_carry_rows += tot_rows;
    }
    __syncthreads();
  }

  if (threadIdx.x == 0) {
    int e = s_err;
    if (e == 0 && (s_carry_rows != s_local || s_carry_segs > max_segs)) e = CP_ERR_METADATA;
    s_err = e;
    hdr->magic = kMetaMagic;
    hdr->status = e;
    hdr->strategy = strategy;
    hdr->cp_size = cp;
    hdr->rank = rank;
    hdr->n_docs = n_docs;
    hdr->s_local = s_local;
    hdr->n_segs = e ? 0 : s_carry_segs;
    hdr->valid_end = s_valid_end;
    hdr->pad_between_seqs = pad;
    hdr->total_tokens = T;
    hdr->max_segs = max_segs;
    hdr->seg_offset = (int32_t)seg_offset_bytes();
    hdr->rows_offset = (int32_t)rows_offset_bytes(n_docs);
    hdr->lists_offset = (int32_t)lists_offset_bytes(n_docs, s_local);
    hdr->n_kblocks = (int32_t)n_tiles_of(T);
    if (e) atomicCAS(&g_status_partition, 0, e);
  }
  __syncthreads();
  if (s_err) return;

  // pass 2: per-row tables, one warp per segment
  const int n_segs = s_carry_segs;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int k = warp; k < n_segs; k += kThreads / 32) {
    const Segment s = segs[k];
    for (int u = lane; u < s.len; u += 32) {
      const int t = s.local_start + u;
      const int g = s.global_start + u;
      const bool valid = u < s.valid_len;
      idx[t] = g;
      if (restore) restore[g] = R0 + t;
      row_lo[t] = valid ? s.doc_lo : 0;
      row_hi[t] = valid ? g : -1;
    }
  }

  // pass 3: block lists (from the segment table written above); each list's
  // block count is also kept in shared memory when both families fit
  __syncthreads();
  const MetaView mv = meta_view(meta);
  const int n_qt = (int)n_tiles_of(s_local);
  const int n_kb = (int)n_tiles_of(T);
  const bool counts_in_smem = n_qt + n_kb <= kNbCap;
  int2* lists = reinterpret_cast<int2*>(meta + lists_offset_bytes(n_docs, s_local));
  for (int q = threadIdx.x; q < n_qt + n_kb; q += kThreads) {
    int2* out = lists + (kListBytes / 8) * q;
    int cnt;
    if (q < n_qt) {
      const int t0 = q * kTile;
      cnt = build_kv_intervals(mv, t0, min(kTile, s_local - t0), kTile, out + 1, kListCap);
    } else {
      const int j0 = (q - n_qt) * kTile;
      cnt = build_q_intervals(mv, j0, min(j0 + kTile, T) - 1, kTile, out + 1, kListCap);
    }
    int nb = 0;
    for (int i = 0; i < min(cnt, kListCap); ++i) nb += out[1 + i].y - out[1 + i].x + 1;
    out[0] = make_int2(cnt, nb);
    if (counts_in_smem) s_nb[q] = nb;
  }

  // pass 4: heaviest-first work order of each list family
  __syncthreads();
  build_work_order(lists, n_qt, n_kb, s_nb, counts_in_smem);
}

// ---------------------------------------------------------------------------
// P2P ring metadata ("THD P2P context-parallel regression ...", §Describe the
// bug: the per-step sequence metadata of the ring comm type).  At ring step i
// rank r holds the K/V shard of rank j = (r - i) mod cp; its attention is a
// cp_size = 1 call of the rank's s_local queries against that shard's s_local
// keys, with every query row's visible keys one contiguous range of the
// shard's local rows: DUAL_CHUNK_SWAP keeps a document's two chunks adjacent
// and in global order in every rank's layout, NO_LOAD_BALANCE shards are
// contiguous.  One CTA per step writes that step's metadata block (all steps
// of a rank in one launch): row tables in shard-local key coordinates, block
// lists and the work order; the segment table is not used (n_segs = 0) and
// its area holds the per-document local offsets while the block is built.
__global__ void __launch_bounds__(kThreads, 1)
p2p_index_kernel(const int32_t* __restrict__ cu, const int32_t* __restrict__ cup, int n_docs,
                 int T, int cp, int rank, int strategy, int pad, char* __restrict__ meta_base,
                 size_t step_bytes) {
  __shared__ int s_warp[32];
  __shared__ int s_err;
  __shared__ int s_carry;
  __shared__ int s_nb[kNbCap];
  const int step = blockIdx.x;
  const int j = ((rank - step) % cp + cp) % cp;  // owner of the K/V shard held at this step
  char* meta = meta_base + (size_t)step * step_bytes;
  MetaHeader* hdr = reinterpret_cast<MetaHeader*>(meta);
  const int s_local = T / cp;
  int32_t* doc_off = reinterpret_cast<int32_t*>(meta + seg_offset_bytes());  // [n_docs + 1]
  int32_t* row_lo = reinterpret_cast<int32_t*>(meta + rows_offset_bytes(n_docs));
  int32_t* row_hi = row_lo + s_local;
  const bool dcs = strategy == CP_DUAL_CHUNK_SWAP;

  if (threadIdx.x == 0) {
    int e = 0;
    if (cup[0] != 0 || cup[n_docs] != T) e = CP_ERR_METADATA;
    if (pad && cu[0] != 0) e = CP_ERR_METADATA;
    s_err = e;
    s_carry = 0;
  }
  __syncthreads();
  // per-document local offset of DUAL_CHUNK_SWAP (2*c_d rows per document on
  // every rank), and checks
  for (int base = 0; base < n_docs; base += kThreads) {
    const int d = base + threadIdx.x;
    int rows = 0;
    if (d < n_docs) {
      const int P = cup[d + 1] - cup[d];
      const int L = pad ? (cu[d + 1] - cu[d]) : P;
      if (P < 0 || L < 0 || L > P) atomicCAS(&s_err, 0, CP_ERR_METADATA);
      if (dcs && P > 0 && P % (2 * cp)) atomicCAS(&s_err, 0, CP_ERR_DIVISIBILITY);
      rows = dcs ? 2 * (P / (2 * cp)) : 0;
    }
    int tot;
    const int off = block_exclusive_scan(rows, s_warp, &tot) + s_carry;
    if (d < n_docs) doc_off[d] = off;
    __syncthreads();
    if (threadIdx.x == 0) s_carry += tot;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    doc_off[n_docs] = s_carry;
    int e = s_err;
    if (e == 0 && dcs && s_carry != s_local) e = CP_ERR_METADATA;
    s_err = e;
    hdr->magic = kMetaMagic;
    hdr->status = e;
    hdr->strategy = strategy;
    hdr->cp_size = 1;
    hdr->rank = 0;
    hdr->n_docs = n_docs;
    hdr->s_local = s_local;
    hdr->n_segs = 0;
    hdr->valid_end = 0;
    hdr->pad_between_seqs = pad;
    hdr->total_tokens = s_local;
    hdr->max_segs = max_segs_for(n_docs);
    hdr->seg_offset = (int32_t)seg_offset_bytes();
    hdr->rows_offset = (int32_t)rows_offset_bytes(n_docs);
    hdr->lists_offset = (int32_t)lists_offset_bytes(n_docs, s_local);
    hdr->n_kblocks = (int32_t)n_tiles_of(s_local);
    if (e) atomicCAS(&g_status_partition, 0, e);
  }
  __syncthreads();
  if (s_err) return;

  // row tables: keys of the held shard each local query row sees
  for (int t = threadIdx.x; t < s_local; t += kThreads) {
    int d, g;
    if (dcs) {  // last document whose local range starts at or before t
      int a = 0, b = n_docs - 1;
      while (a < b) {
        const int mid = (a + b + 1) >> 1;
        if (doc_off[mid] <= t) a = mid; else b = mid - 1;
      }
      d = a;
      while (d + 1 < n_docs && doc_off[d + 1] <= t) ++d;  // skip empty documents
      const int c = (cup[d + 1] - cup[d]) / (2 * cp);
      const int u = t - doc_off[d];
      g = cup[d] + (u < c ? rank * c + u : (2 * cp - 1 - rank) * c + (u - c));
    } else {
      g = rank * s_local + t;
      int a = 0, b = n_docs - 1;  // last document with cup[d] <= g
      while (a < b) {
        const int mid = (a + b + 1) >> 1;
        if (cup[mid] <= g) a = mid; else b = mid - 1;
      }
      d = a;
      while (d + 1 < n_docs && cup[d + 1] <= g) ++d;
    }
    const int L = pad ? (cu[d + 1] - cu[d]) : (cup[d + 1] - cup[d]);
    int lo = 0, cnt = 0;
    if (g < cup[d] + L) {
      if (dcs) {
        const int c = (cup[d + 1] - cup[d]) / (2 * cp);
        lo = doc_off[d];
        cnt = clampi(g - (cup[d] + j * c) + 1, 0, c) +
              clampi(g - (cup[d] + (2 * cp - 1 - j) * c) + 1, 0, c);
      } else {
        const int a = max(cup[d], j * s_local), b = min(cup[d + 1], (j + 1) * s_local);
        if (b > a) {
          lo = a - j * s_local;
          cnt = clampi(g - a + 1, 0, b - a);
        }
      }
    }
    row_lo[t] = cnt > 0 ? lo : 0;
    row_hi[t] = cnt > 0 ? lo + cnt - 1 : -1;
  }
  __syncthreads();

  // block lists: per query tile the key blocks its rows see (rows come in
  // document order, so their block ranges arrive sorted by start), then per
  // key block the query tiles seeing it
  const int n_qt = (int)n_tiles_of(s_local);
  const int n_kb = n_qt;
  const bool counts_in_smem = n_qt + n_kb <= kNbCap;
  int2* lists = reinterpret_cast<int2*>(meta + lists_offset_bytes(n_docs, s_local));
  for (int q = threadIdx.x; q < n_qt; q += kThreads) {
    int2* out = lists + (kListBytes / 8) * q;
    int cnt = 0, cur_lo = 0, cur_hi = -2;
    for (int t = q * kTile; t < min(s_local, (q + 1) * kTile); ++t) {
      if (row_hi[t] < 0) continue;
      const int blo = row_lo[t] / kTile, bhi = row_hi[t] / kTile;
      if (cur_hi >= -1 && blo <= cur_hi + 1) {
        cur_hi = max(cur_hi, bhi);
        cur_lo = min(cur_lo, blo);
      } else {
        if (cur_hi >= -1) {
          if (cnt < kListCap) out[1 + cnt++] = make_int2(cur_lo, cur_hi);
          else out[kListCap] = make_int2(out[kListCap].x, cur_hi);  // over capacity: widen the last
        }
        cur_lo = blo;
        cur_hi = bhi;
      }
    }
    if (cur_hi >= -1) {
      if (cnt < kListCap) out[1 + cnt++] = make_int2(cur_lo, cur_hi);
      else out[kListCap] = make_int2(out[kListCap].x, max(out[kListCap].y, cur_hi));
    }
    int nb = 0;
    for (int i = 0; i < cnt; ++i) nb += out[1 + i].y - out[1 + i].x + 1;
    out[0] = make_int2(cnt, nb);
    if (counts_in_smem) s_nb[q] = nb;
  }
  __syncthreads();
  for (int kb = threadIdx.x; kb < n_kb; kb += kThreads) {
    int2* out = lists + (kListBytes / 8) * (n_qt + kb);
    int cnt = 0, cur_lo = -1, cur_hi = -2;
    for (int q = 0; q < n_qt; ++q) {
      const int2* l = lists + (kListBytes / 8) * q;
      const int n = min(l[0].x, kListCap);
      bool hit = false;
      for (int i = 0; i < n && !hit; ++i) hit = l[1 + i].x <= kb && kb <= l[1 + i].y;
      if (!hit) continue;
      if (q == cur_hi + 1) {
        cur_hi = q;
      } else {
        if (cur_lo >= 0) {
          if (cnt < kListCap) out[1 + cnt++] = make_int2(cur_lo, cur_hi);
          else out[kListCap] = make_int2(out[kListCap].x, cur_hi);
        }
        cur_lo = cur_hi = q;
      }
    }
    if (cur_lo >= 0) {
      if (cnt < kListCap) out[1 + cnt++] = make_int2(cur_lo, cur_hi);
      else out[kListCap] = make_int2(out[kListCap].x, max(out[kListCap].y, cur_hi));
    }
    int nb = 0;
    for (int i = 0; i < cnt; ++i) nb += out[1 + i].y - out[1 + i].x + 1;
    out[0] = make_int2(cnt, nb);
    if (counts_in_smem) s_nb[n_qt + kb] = nb;
  }
  __syncthreads();
  build_work_order(lists, n_qt, n_kb, s_nb, counts_in_smem);
}

}  // namespace
}  // namespace cpthd

using namespace cpthd;

extern "C" size_t cp_meta_bytes(int n_docs, int64_t total_tokens, int cp_size) {
  if (n_docs < 0 || total_tokens < 0 || cp_size < 1 || total_tokens % cp_size) return 0;
  return meta_bytes_for(n_docs, total_tokens / cp_size, cp_size);
}

extern "C" int cp_partition_index(const int32_t* d_cu, const int32_t* d_cup, int n_docs,
                                  int64_t total_tokens, int cp_size, int rank,
                                  cp_strategy_t strategy, int pad_between_seqs, int32_t* d_idx,
                                  int32_t* d_restore, void* d_meta, size_t meta_bytes,
                                  void* stream) {
  if (!d_cup || !d_idx || !d_meta) return CP_ERR_INVALID_ARG;
  if (pad_between_seqs && !d_cu) return CP_ERR_INVALID_ARG;
  if (n_docs < 1 || cp_size < 1 || rank < 0 || rank >= cp_size) return CP_ERR_INVALID_ARG;
  if (strategy != CP_DUAL_CHUNK_SWAP && strategy != CP_NO_LOAD_BALANCE) return CP_ERR_INVALID_ARG;
  if (total_tokens < 0 || total_tokens > INT32_MAX) return CP_ERR_INVALID_ARG;
  if (total_tokens % cp_size) return CP_ERR_DIVISIBILITY;
  const int64_t s_local = total_tokens / cp_size;
  if (meta_bytes < meta_bytes_for(n_docs, s_local, cp_size)) return CP_ERR_WORKSPACE;
  if (!cpthd_host::aligned16(d_meta)) return CP_ERR_ALIGNMENT;
  partition_kernel<<<1, 1024, 0, cpthd_host::as_stream(stream)>>>(
      d_cu, d_cup, n_docs, (int)total_tokens, cp_size, rank, (int)strategy,
      pad_between_seqs ? 1 : 0, d_idx, d_restore, reinterpret_cast<char*>(d_meta), 0);
  return cpthd_host::launch_status();
}

extern "C" int cp_partition_index_all(const int32_t* d_cu, const int32_t* d_cup, int n_docs,
                                      int64_t total_tokens, int cp_size, cp_strategy_t strategy,
                                      int pad_between_seqs, int32_t* d_idx_all,
                                      int32_t* d_restore, void* d_meta, size_t meta_stride,
                                      void* stream) {
  if (!d_cup || !d_idx_all || !d_meta) return CP_ERR_INVALID_ARG;
  if (pad_between_seqs && !d_cu) return CP_ERR_INVALID_ARG;
  if (n_docs < 1 || cp_size < 1 || cp_size > 65535) return CP_ERR_INVALID_ARG;
  if (strategy != CP_DUAL_CHUNK_SWAP && strategy != CP_NO_LOAD_BALANCE) return CP_ERR_INVALID_ARG;
  if (total_tokens < 0 || total_tokens > INT32_MAX) return CP_ERR_INVALID_ARG;
  if (total_tokens % cp_size) return CP_ERR_DIVISIBILITY;
  const int64_t s_local = total_tokens / cp_size;
  if (meta_stride < meta_bytes_for(n_docs, s_local, cp_size)) return CP_ERR_WORKSPACE;
  if (!cpthd_host::aligned16(d_meta) || (meta_stride & 15)) return CP_ERR_ALIGNMENT;
  partition_kernel<<<cp_size, 1024, 0, cpthd_host::as_stream(stream)>>>(
      d_cu, d_cup, n_docs, (int)total_tokens, cp_size, 0, (int)strategy,
      pad_between_seqs ? 1 : 0, d_idx_all, d_restore, reinterpret_cast<char*>(d_meta),
      meta_stride);
  return cpthd_host::launch_status();
}


extern "C" size_t cp_p2p_meta_bytes(int n_docs, int64_t total_tokens, int cp_size) {
  if (n_docs < 0 || total_tokens < 0 || cp_size < 1 || total_tokens % cp_size) return 0;
  const int64_t s_local = total_tokens / cp_size;
  return (meta_bytes_for(n_docs, s_local, 1) + 15) & ~(size_t)15;
}

extern "C" int cp_p2p_index(const int32_t* d_cu, const int32_t* d_cup, int n_docs,
                            int64_t total_tokens, int cp_size, int rank, cp_strategy_t strategy,
                            int pad_between_seqs, void* d_meta, size_t meta_bytes, void* stream) {
  if (!d_cup || !d_meta) return CP_ERR_INVALID_ARG;
  if (pad_between_seqs && !d_cu) return CP_ERR_INVALID_ARG;
  if (n_docs < 1 || cp_size < 1 || rank < 0 || rank >= cp_size) return CP_ERR_INVALID_ARG;
  if (strategy != CP_DUAL_CHUNK_SWAP && strategy != CP_NO_LOAD_BALANCE) return CP_ERR_INVALID_ARG;
  if (total_tokens < 0 || total_tokens > INT32_MAX) return CP_ERR_INVALID_ARG;
  if (total_tokens % cp_size) return CP_ERR_DIVISIBILITY;
  const size_t step = cp_p2p_meta_bytes(n_docs, total_tokens, cp_size);
  if (meta_bytes < step * (size_t)cp_size) return CP_ERR_WORKSPACE;
  if (!cpthd_host::aligned16(d_meta)) return CP_ERR_ALIGNMENT;
  p2p_index_kernel<<<cp_size, kThreads, 0, cpthd_host::as_stream(stream)>>>(
      d_cu, d_cup, n_docs, (int)total_tokens, cp_size, rank, (int)strategy,
      pad_between_seqs ? 1 : 0, reinterpret_cast<char*>(d_meta), step);
  return cpthd_host::launch_status();
}

extern "C" int cpthd_status_partition(int reset) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status_partition, sizeof(int)) != cudaSuccess) return CP_ERR_CUDA;
  if (reset) {
    int z = 0;
    if (cudaMemcpyToSymbol(g_status_partition, &z, sizeof(int)) != cudaSuccess) return CP_ERR_CUDA;
  }
  return v;
}
