// attn_bwd_tc.cu -- causal varlen attention backward of one CP rank on the
// Blackwell tensor cores (tcgen05 + TMEM + TMA), built for sm_103a.
//
// The tensor-core operands are all bf16 or all fp16 (F16).  With bf16, the
// probabilities P and dS go into the products as two bf16 terms each (the
// rounded value and its rounding remainder: one extra product each), which
// carries them to about 16 bits; fp16 (11 bits) needs one term.
//
// The backward of the forward in attn_fwd_tc.cu ("[PyTorch] Add
// no-load-balance THD all-gather CP", §What changed: backward uses the
// forward's token layout): with Delta_t = dO_t . O_t (attn_delta),
//   P = exp(scale q.k - LSE), dS = P (dO.v - Delta),
//   dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO.
// Two persistent kernels (one CTA per SM walking a static list of work
// items, all barrier phases on global counters so the pipeline carries
// across items), no atomics (bitwise deterministic):
//
// attn_dq_tc   items (128-query tile, head), iterating the key blocks the
//              tile attends.  S = Q K^T and dP = dO V^T into TMEM (M=128
//              queries, N=128 keys); the compute warps form dS into TMEM
//              columns of its own; dQ += dS K with A = dS from TMEM, B = K as
//              an MN-major operand.  K tiles sit in a 3-stage ring
//              (released after dQ), V tiles in a 2-stage ring (released after
//              dP).
// attn_dkdv_tc items (128-key block, head), iterating the rank's query tiles
//              that attend the block (precomputed block lists).  S^T = K Q^T
//              and dP^T = V dO^T into TMEM (M=128 keys, N=128 queries); the
//              compute warps form P^T and dS^T in TMEM over S^T and dP^T;
//              dV += P^T dO and dK += dS^T Q (A from TMEM, B = dO / Q as
//              MN-major operands).  Each item's partial dK/dV are added into
//              the caller's fp32 accumulators by the item's only owner, with
//              bulk tensor reduce-adds of staged 32 x 32 chunks (one add per
//              element per launch, so the sums are still bitwise
//              reproducible).
// Warp roles: warps 0-7 compute (warp w serves TMEM lanes 32*(w%4).. and the
// column half w/4 of every row, so two warps share each row's elementwise
// work), warp 8 TMA producer, warp 9 TMEM allocator + single-thread MMA
// issuer.  The MMA thread interleaves consecutive steps (a step's products are
// issued while the previous step's gradient product is still pending) so the
// tensor core keeps working while the compute warps run the elementwise part.  A compute
// thread writes P / dS back only into TMEM columns it has itself already read,
// so the two column halves never race.  Every wait is bounded.
#include <math.h>

#include "common.cuh"
#include "sm100.cuh"
#include "tma_host.cuh"

namespace cpthd {

static __device__ int g_status_bwd_tc;

namespace {

using namespace sm100;
using bf16 = __nv_bfloat16;

constexpr int kThr = 320;
constexpr int kCompute = 256;  // threads of warps 0-7
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr int kBox = 128 * 128;  // one 128-row x 128-byte TMA box
constexpr uint32_t kCols = 512;
constexpr uint64_t kLimitNs = 4000000000ull;
constexpr float kLog2ef = 1.4426950408889634f;

struct BwdArgs {
  const float* lse;    // [H, s_local]
  const float* delta;  // [H, s_local]
  void* dq;            // [s_local, H, D]: bf16, or fp32 when dq_mode != 0
  float* dk;           // [T, H, D]
  float* dv;
  const void* meta;
  size_t meta_bytes;
  int T, H, s_local, cp, rank, strategy;
  float scale, scale_log2;
  int store;    // dK/dV partials stored (every row written) instead of added
  int dq_mode;  // 0: dQ stored as bf16; 1: stored as fp32; 2: added into fp32
  // rank-grouped dK/dV (attn_dkdv_tc only): n_ranks > 1 walks, for every key
  // block, the attending query tiles of all n_ranks ranks.  Then meta is rank
  // 0's metadata and rank r's lies meta_stride bytes further per rank; Q / dO
  // are the rank-concatenated [n_ranks * s_local, H, D] buffers; lse and delta
  // are [n_ranks][H][s_local]; gorder is the key blocks' heaviest-first order
  // by their total over the ranks.
  int n_ranks;
  int64_t meta_stride;
  const int2* gorder;
  int* gorder_tot;  // n ints of scratch for the order's totals
  // ring mode: the P2P ring's steps in one pass.  dQ (n_steps > 1, or
  // ring_cp > 0): rank ring_rank's n_steps steps, step i's metadata
  // (cp_size = 1) step_stride bytes after meta, its keys the shard of rank
  // (ring_rank - i) mod ring_cp, rows s_local * that rank of the K / V
  // tensors; gorder is then the rank's query tiles heaviest first by their
  // count over the steps.  dK/dV (ring = 1, n_ranks = ring_cp): items are the
  // key blocks of every shard; the ranks' step metadata lie meta_stride bytes
  // apart from meta; rank r reads shard j at its step (r - j) mod ring_cp;
  // dK / dV rows are rank-concatenated.
  int ring, n_steps, ring_rank, ring_cp;
  int64_t step_stride;
  // rank-grouped dK/dV with the reduce-scatter's scatter fused in (rs = 1):
  // the summed dK / dV of global key row j go, rounded to bf16, to row
  // rs_row[j] (j when rs_row is null) of the rank-concatenated dk16 / dv16
  // [T, H, D] instead of the fp32 dk / dv.
  int rs;
  const int32_t* rs_row;
  uint16_t* dk16;
  uint16_t* dv16;
};

// Metadata of ring step i of the dQ pass (step 0 outside ring mode).
__device__ __forceinline__ const void* step_meta(const BwdArgs& a, int i) {
  return reinterpret_cast<const char*>(a.meta) + a.step_stride * i;
}

// Ring steps of rank r: every step for DUAL_CHUNK_SWAP, steps 0..r for
// NO_LOAD_BALANCE (later ranks' shards hold only later tokens).
__device__ __forceinline__ int ring_steps_of(const BwdArgs& a, int r) {
  return a.strategy == (int)CP_NO_LOAD_BALANCE ? min(r + 1, a.ring_cp) : a.ring_cp;
}

// Source s of a rank-grouped dK/dV item on key shard j: its metadata, or null
// when the source has no step for that shard (ring mode).  Outside ring mode
// the source is rank s; in ring mode rank s at its step (s - j) mod ring_cp.
__device__ __forceinline__ const void* kv_source(const BwdArgs& a, int shard, int src) {
  if (!a.ring) return reinterpret_cast<const char*>(a.meta) + a.meta_stride * src;
  const int i = (src - shard + a.ring_cp) % a.ring_cp;
  if (i >= ring_steps_of(a, src)) return nullptr;
  return reinterpret_cast<const char*>(a.meta) + a.meta_stride * src + a.step_stride * i;
}

// Destination row of key row kr under the fused scatter: rs_row[kr] (kr
// without an index); -1 for a row at or past row_end (the end of the item's
// rows), or an index entry outside the output's rows (T; ring mode: the
// ranks' shards, ring_cp * s_local), which also sets the status word.
__device__ __forceinline__ int64_t rs_dst_row(const BwdArgs& a, int kr, int row_end) {
  if (kr >= row_end) return -1;
  const int n = a.ring ? a.ring_cp * a.s_local : a.T;
  const int t = a.rs_row ? __ldg(a.rs_row + kr) : kr;
  if (t < 0 || t >= n) {
    atomicCAS(&g_status_bwd_tc, 0, (int)CP_ERR_INVALID_ARG);
    return -1;
  }
  return t;
}

__device__ __forceinline__ bool meta_ok_bwd(const BwdArgs& a, const MetaHeader* h) {
  const bool ok = meta_matches(h, a.meta_bytes, a.T, a.s_local, a.cp, a.rank, a.strategy);
  if (!ok && threadIdx.x == 0)
    atomicCAS(&g_status_bwd_tc, 0, h->status != 0 ? h->status : (int)CP_ERR_METADATA);
  return ok;
}

// Metadata of rank r of a rank-grouped call.
__device__ __forceinline__ const void* rank_meta(const BwdArgs& a, int r) {
  return reinterpret_cast<const char*>(a.meta) + a.meta_stride * r;
}

// Every rank's metadata of a rank-grouped call matches (rank r at r); in ring
// mode every step metadata the call reads (cp_size = 1, rank 0).
__device__ __forceinline__ bool meta_ok_grouped(const BwdArgs& a) {
  bool ok = true;
  int bad = 0;
  if (a.ring) {
    for (int r = 0; r < a.n_ranks && ok; ++r)
      for (int i = 0; i < ring_steps_of(a, r) && ok; ++i) {
        const MetaHeader* h = reinterpret_cast<const MetaHeader*>(
            reinterpret_cast<const char*>(a.meta) + a.meta_stride * r + a.step_stride * i);
        ok = meta_matches(h, (size_t)a.meta_bytes, a.T, a.s_local, a.cp, a.rank, a.strategy);
        if (!ok) bad = h->status != 0 ? h->status : (int)CP_ERR_METADATA;
      }
  } else {
    for (int r = 0; r < a.n_ranks && ok; ++r) {
      const MetaHeader* h = reinterpret_cast<const MetaHeader*>(rank_meta(a, r));
      ok = meta_matches(h, (size_t)a.meta_stride, a.T, a.s_local, a.cp, r, a.strategy);
      if (!ok) bad = h->status != 0 ? h->status : (int)CP_ERR_METADATA;
    }
  }
  if (!ok && threadIdx.x == 0) atomicCAS(&g_status_bwd_tc, 0, bad);
  return ok;
}

// Every ring step's metadata of a dQ ring pass matches (cp_size = 1, rank 0).
__device__ __forceinline__ bool meta_ok_steps(const BwdArgs& a) {
  bool ok = true;
  int bad = 0;
  for (int i = 0; i < a.n_steps && ok; ++i) {
    const MetaHeader* h = reinterpret_cast<const MetaHeader*>(step_meta(a, i));
    ok = meta_matches(h, a.meta_bytes, a.T, a.s_local, a.cp, a.rank, a.strategy);
    if (!ok) bad = h->status != 0 ? h->status : (int)CP_ERR_METADATA;
  }
  if (!ok && threadIdx.x == 0) atomicCAS(&g_status_bwd_tc, 0, bad);
  return ok;
}

__device__ __forceinline__ void fail(volatile int* abort) {
  *abort = 1;
  atomicCAS(&g_status_bwd_tc, 0, (int)CP_ERR_TIMEOUT);
}

struct Iter {  // flattened walk over an item's block intervals
  const int2* iv;
  int n, i, b;
  __device__ void init(const int2* p, int cnt) { iv = p; n = cnt; i = 0; b = cnt > 0 ? p[0].x : 0; }
  __device__ void next() {
    if (i < n && b < iv[i].y) {
      ++b;
    } else {
      ++i;
      if (i < n) b = iv[i].x;
    }
  }
};

// Work-item order (item_of): dQ takes its query tiles heaviest first over all
// heads, like the forward; dK/dV one head at a time, so that the head's
// streamed Q / dO tiles stay resident in L2 across its key blocks (measured
// on the 65536-token, 32-head workload: about 5% less backward time than
// heaviest first over all heads for dK/dV, about 1.5% more with dQ also taken
// one head at a time).
constexpr int kDqHeadGroup = 1 << 20, kKvHeadGroup = 1;

// One work item: a 128-row tile (dQ: query tile; dK/dV: key block), a head,
// and the blocks of the tile's precomputed list.
struct Item {
  const int2* list;  // the tile's block list: count in list[0].x, intervals in list[1..]
  int tile, h, nb;
  int shard = 0;  // ring-mode dK/dV: the key shard of block `tile`
  // item k: the q-th heaviest tile of head h, heads in groups of G (item_of)
  __device__ void load(const int2* order, const int2* lists, int k, int H, int n_tiles, int G) {
    int q;
    item_of(k, n_tiles, H, G, &q, &h);
    const int2 o = order[min(max(q, 0), n_tiles - 1)];  // that tile and its block count
    tile = min(max(o.x, 0), n_tiles - 1);
    list = lists + (kListBytes / 8) * tile;
    nb = o.y;
  }
  __device__ int n_iv() const { return min(list[0].x, kListCap); }
};

// A dK/dV work item: key block `tile`, head h, and its number of query-tile
// steps -- in a rank-grouped call the sum of every rank's count for the block
// (each rank's block list header) that the ordering kernel stored with it;
// the producer walks the same headers rank by rank.
__device__ __forceinline__ Item kv_item(const BwdArgs& a, const MetaView& m, int k, int n_kb) {
  Item it;
  if (a.n_ranks <= 1) {
    it.load(m.korder, m.klists, k, a.H, n_kb, kKvHeadGroup);
    return it;
  }
  int q;
  item_of(k, n_kb, a.H, kKvHeadGroup, &q, &it.h);  // as Item::load
  const int2 o = a.gorder[min(max(q, 0), n_kb - 1)];
  const int x = min(max(o.x, 0), n_kb - 1);
  if (a.ring) {  // every shard's blocks: x = shard * (blocks per shard) + block
    const int per = (int)n_tiles_of(a.s_local);
    it.shard = x / per;
    it.tile = x % per;
  } else {
    it.tile = x;
  }
  it.list = nullptr;
  it.nb = o.y;  // the sum over the ranks (steps), formed by the ordering kernel
  return it;
}

// The step count of dK/dV item k alone (what the MMA warp needs of it).
__device__ __forceinline__ int kv_item_nb(const BwdArgs& a, const MetaView& m, int k, int n_kb) {
  int q, h;
  item_of(k, n_kb, a.H, kKvHeadGroup, &q, &h);
  return (a.n_ranks > 1 ? a.gorder : m.korder)[min(max(q, 0), n_kb - 1)].y;
}

// dQ work item: outside ring mode as Item::load; in ring mode the q-th
// heaviest of the rank's query tiles by their count over the ring steps.
__device__ __forceinline__ Item dq_item(const BwdArgs& a, const MetaView& m, int k, int n_qt) {
  Item it;
  if (a.n_steps <= 1) {
    it.load(m.qorder, m.qlists, k, a.H, n_qt, kDqHeadGroup);
    return it;
  }
  int q;
  item_of(k, n_qt, a.H, kDqHeadGroup, &q, &it.h);
  const int2 o = a.gorder[min(max(q, 0), n_qt - 1)];
  it.tile = min(max(o.x, 0), n_qt - 1);
  it.list = nullptr;
  it.nb = o.y;
  return it;
}

// The key blocks of a dQ item in order: the tile's block list, or in ring mode
// the lists of the rank's ring steps one after another (the steps with
// blocks), each step's blocks in its shard; b is a block of the current step's
// shard, kv_off the shard's first row in the K / V tensors, step the step.
struct BwdWalk {
  const BwdArgs* a;
  Iter bi;
  int tile, step, left, kv_off;
  __device__ void init(const BwdArgs& args, int t) {
    a = &args;
    tile = t;
    step = -1;
    left = 0;
    kv_off = 0;
    advance();
  }
  __device__ void advance() {
    const int n = a->n_steps > 1 ? a->n_steps : 1;
    while (left == 0 && step + 1 < n) {
      ++step;
      const int2* list = meta_view(step_meta(*a, step)).qlists + (kListBytes / 8) * tile;
      left = list[0].y;
      bi.init(list + 1, min(list[0].x, kListCap));
      kv_off = a->ring_cp > 0
                   ? ((a->ring_rank - step + a->ring_cp) % a->ring_cp) * a->s_local
                   : 0;
    }
  }
  __device__ int b() const { return bi.b; }
  __device__ void next() {
    --left;
    bi.next();
    if (left == 0) advance();
  }
};

__device__ __forceinline__ uint32_t bar_addr(uint64_t& b) { return smem_u32(&b); }

// K-major operand offset of k-step kk (16 elements) inside a tile of
// 64-element (128-byte) boxes of 128 rows.
__device__ __forceinline__ uint32_t kmajor_off(int kk) { return (kk >> 2) * kBox + (kk & 3) * 32; }

// TMEM column of k-step kk (16 elements) of an A operand written by the two
// column halves: elements [0,64) at columns [0,32), [64,128) at [64,96).
__device__ __forceinline__ uint32_t ts_col(int kk) { return (kk >> 2) * 64 + (kk & 3) * 8; }

// Two-term (hi, lo) bf16 A operands written chunk by chunk over fp32 columns
// that were read first: each half's 64 elements arrive as two chunks of 32,
// chunk c of half h read from columns [64h + 32c, 64h + 32c + 32) and
// written back as its rounded values (16 columns) followed by their rounding
// remainders (16 columns).  Column of the rounded part of k-step kk; the
// remainder is 16 columns further.
__device__ __forceinline__ uint32_t hilo_col(int kk) {
  return (kk >> 2) * 64 + ((kk >> 1) & 1) * 32 + (kk & 1) * 8;
}

// Rounds 32 fp32 values to bf16 pairs and keeps the rounding remainders as a
// second set of bf16 pairs: hi + lo carries about 16 significant bits.
__device__ __forceinline__ void split_bf16(const float* x, uint32_t* hi, uint32_t* lo) {
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    hi[e] = pack_bf16(x[2 * e], x[2 * e + 1]);
    lo[e] = pack_bf16(x[2 * e] - bf16_lo_f(hi[e]), x[2 * e + 1] - bf16_hi_f(hi[e]));
  }
}

// 32 fp32 values -> TMEM columns [col, col+16) as an A operand: fp16 pairs
// (F16), or bf16 pairs followed by the bf16 pairs of their rounding
// remainders at [col+16, col+32) (two bf16 terms carry about 16 significant
// bits; fp16 alone carries 11).
template <bool F16>
__device__ __forceinline__ void store_operand(uint32_t col, const float* x) {
  uint32_t hi[16];
  if (F16) {
#pragma unroll
    for (int e = 0; e < 16; ++e) hi[e] = pack_f16(x[2 * e], x[2 * e + 1]);
    tmem_st16(col, hi);
  } else {
    uint32_t lo[16];
    split_bf16(x, hi, lo);
    tmem_st16(col, hi);
    tmem_st16(col + 16, lo);
  }
}

// p[e] = 2^(p[e] * scl - lse2) for 64 scores (lse2 in the log2 domain, one
// per element pair or shared), the products in paired instructions.
__device__ __forceinline__ void exp2_scores(float* p, uint64_t scl2, const uint64_t* nlse2,
                                            int nlse_stride) {
#pragma unroll
  for (int c2 = 0; c2 < 32; ++c2) {
    float a, b;
    f2_unpack(f2_fma(f2_pack(p[2 * c2], p[2 * c2 + 1]), scl2, nlse2[c2 * nlse_stride]), a, b);
    p[2 * c2] = ex2_approx(a);
    p[2 * c2 + 1] = ex2_approx(b);
  }
}


// ===========================================================================
// dQ
// ===========================================================================
constexpr int kDqKStages = 3;  // K ring (released after dQ)
constexpr int kDqVStages = 2;  // V ring (released after dP)

template <int D>
struct DqLayout {
  static constexpr int TILE = (D / 64) * kBox;
  static constexpr int Q = 0;
  static constexpr int DO = TILE;
  static constexpr int K = 2 * TILE;
  static constexpr int V = K + kDqKStages * TILE;
  static constexpr int BYTES = V + kDqVStages * TILE;
};

// TMEM of attn_dq_tc: S [0,128), dP [128,256), dQ [256,256+D), dS [384,512)
// (fp16 pairs, or two bf16 terms hi, lo; hilo_col).  dS has columns of its own
// so that dP_g can be computed as soon as dP_{g-1} is in registers, while dS_{g-1}
// is still being formed and read by dQ_{g-1}.

struct DqCtl {
  uint64_t qd_full, qd_free;  // Q/dO of the item landed / all its S, dP products done
  uint64_t k_full[kDqKStages], k_empty[kDqKStages];
  uint64_t v_full[kDqVStages], v_empty[kDqVStages];
  uint64_t s_full, s_free, dp_full, dp_free, ds_full, ds_free, done, mma_done;
  uint32_t tmem;
  int abort;
};

// Per key block g the MMA thread issues dP_g as soon as the compute warps have
// read dP_{g-1} into registers (dp_free), then dQ_{g-1} once dS_{g-1} is in
// TMEM, then S_{g+1} once S_g has been read (s_free).  The compute warps are
// then never waiting for dP: it is computed while they form dS_{g-1} and the
// exponentials of block g.  dS_g is written only after dQ_{g-1} has finished
// reading dS_{g-1} (ds_free).  Every per-block barrier completes once per
// block, and each one's next phase needs a step of its waiter first (dP_{g+1}
// waits for dp_free(g), which the compute warps arrive at after waiting for
// dp_full(g); S_{g+1} waits for s_free(g), after s_full(g); dQ_g waits for
// ds_full(g), which follows the wait for ds_free(g-1)), so a parity wait never
// sees a phase two ahead.
template <int D, bool F16>
__global__ void __launch_bounds__(kThr, 1)
attn_dq_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
           const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
           const __grid_constant__ BwdArgs a) {
  using L = DqLayout<D>;
  constexpr int BOXES = D / 64;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the next launch of the rank-grouped backward (the next rank's dQ, or the
  // dK/dV work order) reads nothing this grid writes: it may start as soon as
  // SMs free up (its CTAs land where this grid's CTAs have finished)
  if (threadIdx.x == 0) pdl_launch_dependents();
  const MetaView m = meta_view(a.meta);
  if (a.n_steps > 1 ? !meta_ok_steps(a) : !meta_ok_bwd(a, m.hdr)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sb = smem_u32(smem_raw);  // tiles need 1024-byte alignment (128B swizzle)
  if (sb & 1023u) {
    if (threadIdx.x == 0) atomicCAS(&g_status_bwd_tc, 0, (int)CP_ERR_UNSUPPORTED);
    return;
  }
  DqCtl& c = *reinterpret_cast<DqCtl*>(smem_raw + L::BYTES);
  volatile int& s_abort = *reinterpret_cast<volatile int*>(&c.abort);
  const int n_qt = (int)n_tiles_of(a.s_local);
  const int n_items = n_qt * a.H;

  if (threadIdx.x == 0) {
    c.abort = 0;
    mbar_init(bar_addr(c.qd_full), 1);
    mbar_init(bar_addr(c.qd_free), 1);
    for (int s = 0; s < kDqKStages; ++s) {
      mbar_init(bar_addr(c.k_full[s]), 1);
      mbar_init(bar_addr(c.k_empty[s]), 1);
    }
    for (int s = 0; s < kDqVStages; ++s) {
      mbar_init(bar_addr(c.v_full[s]), 1);
      mbar_init(bar_addr(c.v_empty[s]), 1);
    }
    mbar_init(bar_addr(c.s_full), 1);
    mbar_init(bar_addr(c.s_free), kCompute);
    mbar_init(bar_addr(c.dp_full), 1);
    mbar_init(bar_addr(c.dp_free), kCompute);
    mbar_init(bar_addr(c.ds_full), kCompute);
    mbar_init(bar_addr(c.ds_free), 1);
    mbar_init(bar_addr(c.done), 1);
    mbar_init(bar_addr(c.mma_done), 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&c.tmem), kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c.tmem;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      int ii = 0, gk = 0, gv = 0;
      bool ok = true;
      for (int j = 0; ok && j * (int)gridDim.x < n_items; ++j) {
        const int k = snake_item(j, blockIdx.x, gridDim.x);
        if (k >= n_items) continue;
        const Item it = dq_item(a, m, k, n_qt);
        if (it.nb == 0) continue;
        // single Q/dO buffer: free once the previous item's S, dP retired
        if (!mbar_wait(bar_addr(c.qd_free), (ii & 1) ^ 1, &s_abort, kLimitNs)) {
          fail(&s_abort);
          break;
        }
        const int t0 = it.tile * 128;
        mbar_arrive_expect_tx(bar_addr(c.qd_full), 2 * L::TILE);
#pragma unroll
        for (int b = 0; b < BOXES; ++b) {
          tma_load_3d(sb + L::Q + b * kBox, &tm_q, bar_addr(c.qd_full), b * 64, it.h, t0);
          tma_load_3d(sb + L::DO + b * kBox, &tm_do, bar_addr(c.qd_full), b * 64, it.h, t0);
        }
        ++ii;
        BwdWalk w;
        w.init(a, it.tile);
        for (int j = 0; j < it.nb; ++j, w.next()) {
          const int key0 = w.kv_off + w.b() * 128;  // the block's first row in K / V
          const int ks = gk % kDqKStages;
          if (!mbar_wait(bar_addr(c.k_empty[ks]), ((gk / kDqKStages) & 1) ^ 1, &s_abort,
                         kLimitNs)) {
            fail(&s_abort);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar_addr(c.k_full[ks]), L::TILE);
#pragma unroll
          for (int b = 0; b < BOXES; ++b)
            tma_load_3d(sb + L::K + ks * L::TILE + b * kBox, &tm_k, bar_addr(c.k_full[ks]),
                        b * 64, it.h, key0);
          ++gk;
          const int vs = gv % kDqVStages;
          if (!mbar_wait(bar_addr(c.v_empty[vs]), ((gv / kDqVStages) & 1) ^ 1, &s_abort,
                         kLimitNs)) {
            fail(&s_abort);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar_addr(c.v_full[vs]), L::TILE);
#pragma unroll
          for (int b = 0; b < BOXES; ++b)
            tma_load_3d(sb + L::V + vs * L::TILE + b * kBox, &tm_v, bar_addr(c.v_full[vs]),
                        b * 64, it.h, key0);
          ++gv;
        }
      }
      // drain: every copy this CTA issued must land before shared memory goes away
      int never = 0;
      if (ii > 0) mbar_wait(bar_addr(c.qd_full), (ii - 1) & 1, &never, kLimitNs);
      for (int j = max(0, gk - kDqKStages); j < gk; ++j)
        mbar_wait(bar_addr(c.k_full[j % kDqKStages]), (j / kDqKStages) & 1, &never, kLimitNs);
      for (int j = max(0, gv - kDqVStages); j < gv; ++j)
        mbar_wait(bar_addr(c.v_full[j % kDqVStages]), (j / kDqVStages) & 1, &never, kLimitNs);
    }
  } else if (warp == kMmaWarp) {
    // The whole warp runs the issue loop (uniform control flow, warp-uniform
    // waits); one elected lane issues each MMA and commit.
    auto wait_w = [&](uint32_t b, uint32_t parity) -> bool {
      const bool w = mbar_wait(b, parity, &s_abort, kLimitNs);
      return __all_sync(0xffffffffu, w);
    };
    {
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false, F16);
      constexpr uint32_t idQ = idesc_bf16_f32(128, D, false, true, F16);
      // operand descriptors at the tiles' first bytes (K-major, and K as MN-major)
      const uint64_t dsc_q = sdesc_sw128(sb + L::Q, 16, 1024);
      const uint64_t dsc_do = sdesc_sw128(sb + L::DO, 16, 1024);
      const uint64_t dsc_k = sdesc_sw128(sb + L::K, 16, 1024);
      const uint64_t dsc_v = sdesc_sw128(sb + L::V, 16, 1024);
      const uint64_t dsc_kmn = sdesc_sw128(sb + L::K, kBox, 1024);
      int ii = 0, g = 0;
      int pend = -1;  // block whose dQ product is still to be issued
      bool pend_first = false;
      // dQ_pend += dS K : A = dS (TMEM, its own columns), B = K tile as
      // MN-major (N = d); bf16 dS is the sum of two terms (rounded values,
      // then their remainders): two products per k-step, fp16 dS one.  An
      // item's first dQ starts afresh: its ds_full comes after the compute
      // warps have read the previous item's dQ out of TMEM.
      auto issue_dq = [&]() -> bool {
        if (!wait_w(bar_addr(c.ds_full), pend & 1)) return false;
        tc_fence_after();
        const int pks = pend % kDqKStages;
        const uint64_t bkm = sdesc_add(dsc_kmn, pks * L::TILE);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t b = sdesc_add(bkm, kk * 2048);
          umma_bf16_ts_w(tmem + 256, tmem + 384 + hilo_col(kk), b, idQ,
                       (!pend_first || kk > 0) ? 1u : 0u);
          if (!F16) umma_bf16_ts_w(tmem + 256, tmem + 384 + hilo_col(kk) + 16, b, idQ, 1u);
        }
        umma_commit_w(bar_addr(c.k_empty[pks]));
        umma_commit_w(bar_addr(c.ds_free));
        return true;
      };
      // S_g = Q K_g^T into TMEM columns [0,128).  S_g overwrites S_{g-1}: the
      // compute warps must have read it (s_free), and K_g must have landed.
      auto issue_s = [&](int gs_) -> bool {
        const int ks = gs_ % kDqKStages;
        if (!wait_w(bar_addr(c.k_full[ks]), (gs_ / kDqKStages) & 1) ||
            (gs_ > 0 && !wait_w(bar_addr(c.s_free), (gs_ - 1) & 1)))
          return false;
        tc_fence_after();
        const uint64_t bk = sdesc_add(dsc_k, ks * L::TILE);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = kmajor_off(kk);
          umma_bf16_w(tmem, sdesc_add(dsc_q, off), sdesc_add(bk, off), idS, kk > 0);
        }
        umma_commit_w(bar_addr(c.s_full));
        return true;
      };
      bool ok = true;
      for (int j = 0; ok && j * (int)gridDim.x < n_items; ++j) {
        const int k = snake_item(j, blockIdx.x, gridDim.x);
        if (k >= n_items) continue;
        const Item it = dq_item(a, m, k, n_qt);
        if (it.nb == 0) continue;
        if (!wait_w(bar_addr(c.qd_full), ii & 1)) {
          fail(&s_abort);
          break;
        }
        ++ii;
        if (!issue_s(g)) {  // the item's first S
          fail(&s_abort);
          break;
        }
        for (int j = 0; j < it.nb; ++j, ++g) {
          const int vs = g % kDqVStages;
          // dP_g = dO V_g^T overwrites dP_{g-1}: the compute warps must have read it
          if ((g > 0 && !wait_w(bar_addr(c.dp_free), (g - 1) & 1)) ||
              !wait_w(bar_addr(c.v_full[vs]), (g / kDqVStages) & 1)) {
            fail(&s_abort);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bv = sdesc_add(dsc_v, vs * L::TILE);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = kmajor_off(kk);
            umma_bf16_w(tmem + 128, sdesc_add(dsc_do, off), sdesc_add(bv, off), idS, kk > 0);
          }
          umma_commit_w(bar_addr(c.dp_full));
          umma_commit_w(bar_addr(c.v_empty[vs]));
          if (j == it.nb - 1) umma_commit_w(bar_addr(c.qd_free));  // every S and dP of the item issued
          if (pend >= 0 && !issue_dq()) {
            fail(&s_abort);
            ok = false;
            break;
          }
          pend = g;
          pend_first = (j == 0);
          if (j + 1 < it.nb && !issue_s(g + 1)) {
            fail(&s_abort);
            ok = false;
            break;
          }
        }
        if (!ok) break;
        // the item's last dQ product, then its epilogue may read dQ
        if (!issue_dq()) {
          fail(&s_abort);
          break;
        }
        pend = -1;
        umma_commit_w(bar_addr(c.done));
      }
      umma_commit_w(bar_addr(c.mma_done));
      int never = 0;
      mbar_wait(bar_addr(c.mma_done), 0, &never, kLimitNs);
    }
  } else {
    const int row = (warp & 3) * 32 + lane;  // TMEM lane = query row of the tile
    const int hf = warp >> 2;                // column half: keys [64hf, 64hf+64)
    const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;
    const float sl2 = a.scale_log2;
    auto wait_warp = [&](uint32_t b, uint32_t parity) -> bool {
      const bool w = mbar_wait(b, parity, &s_abort, kLimitNs);
      return __all_sync(0xffffffffu, w);
    };
    int ii = 0, g = 0;
    bool ok = true;
    for (int j = 0; ok && j * (int)gridDim.x < n_items; ++j) {
      const int k = snake_item(j, blockIdx.x, gridDim.x);
      if (k >= n_items) continue;
      const Item itm = dq_item(a, m, k, n_qt);
      const int t = itm.tile * 128 + row;
      const bool in = t < a.s_local;
      if (itm.nb == 0) {  // no real query row: dQ = 0 (nothing to add in add mode)
        if (in && a.dq_mode == 0) {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<bf16*>(a.dq) +
                                                ((int64_t)t * a.H + itm.h) * D + hf * (D / 2));
#pragma unroll
          for (int q = 0; q < D / 16; ++q) dst[q] = make_uint4(0, 0, 0, 0);
        } else if (in && a.dq_mode == 1) {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<float*>(a.dq) +
                                                ((int64_t)t * a.H + itm.h) * D + hf * (D / 2));
#pragma unroll
          for (int q = 0; q < D / 8; ++q) dst[q] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      int lo = in ? m.row_lo[t] : 0;  // the row's key range (ring mode: per step, below)
      int hi = in ? m.row_hi[t] : -1;
      const float lse2 = hi >= 0 ? a.lse[(int64_t)itm.h * a.s_local + t] * kLog2ef : 0.f;
      const float dl = hi >= 0 ? a.delta[(int64_t)itm.h * a.s_local + t] : 0.f;
      const uint64_t scl2 = f2_pack(sl2, sl2), nlse2 = f2_pack(-lse2, -lse2);
      const uint64_t dl2 = f2_pack(dl, dl);
      BwdWalk w;
      w.init(a, itm.tile);
      int cur_step = 0;  // the ring step whose key range lo / hi hold
      for (int j = 0; j < itm.nb; ++j, w.next(), ++g) {
        if (w.step != cur_step) {  // ring mode: the row's key range in the next step's shard
          const MetaView ms = meta_view(step_meta(a, w.step));
          lo = in ? ms.row_lo[t] : 0;
          hi = in ? ms.row_hi[t] : -1;
          cur_step = w.step;
        }
        if (!wait_warp(bar_addr(c.s_full), g & 1)) {
          fail(&s_abort);
          ok = false;
          break;
        }
        tc_fence_after();
        float p[64];
        tmem_ld32(tmem + lb + 64 * hf, reinterpret_cast<uint32_t*>(p));
        tmem_ld32(tmem + lb + 64 * hf + 32, reinterpret_cast<uint32_t*>(p + 32));
        tc_fence_before();
        mbar_arrive(bar_addr(c.s_free));  // S_{g+1} may now overwrite S
        const int k0 = w.b() * 128 + 64 * hf;  // key (of the step's shard) of this thread's first column
        if (!(lo <= k0 && hi >= k0 + 63)) {  // keys outside the row's range: P = 0
          // (one unsigned compare per column, as in the forward)
          const bool any = hi >= lo;
          const int c_lo = any ? lo - k0 : (1 << 30);
          const unsigned span = any ? (unsigned)(hi - lo) : 0u;
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if ((unsigned)(e - c_lo) > span) p[e] = -INFINITY;
        }
        exp2_scores(p, scl2, &nlse2, 0);
        if (!wait_warp(bar_addr(c.dp_full), g & 1)) {
          fail(&s_abort);
          ok = false;
          break;
        }
        tc_fence_after();
        // dP_g into registers; its columns are then free for dP_{g+1}
        uint32_t dp[64];
        tmem_ld32(tmem + lb + 128 + 64 * hf, dp);
        tmem_ld32(tmem + lb + 128 + 64 * hf + 32, dp + 32);
        tc_fence_before();
        mbar_arrive(bar_addr(c.dp_free));
        // dS = P (dP - Delta)
#pragma unroll
        for (int e2 = 0; e2 < 32; ++e2) {
          float x0, x1;
          f2_unpack(f2_mul(f2_pack(p[2 * e2], p[2 * e2 + 1]),
                           f2_sub(f2_pack(__uint_as_float(dp[2 * e2]),
                                          __uint_as_float(dp[2 * e2 + 1])), dl2)),
                    x0, x1);
          dp[2 * e2] = __float_as_uint(x0);
          dp[2 * e2 + 1] = __float_as_uint(x1);
        }
        // into the dS columns (one fp16 term, or hi and lo bf16 terms), once
        // dQ_{g-1} has finished reading dS_{g-1}
        if (g > 0 && !wait_warp(bar_addr(c.ds_free), (g - 1) & 1)) {
          fail(&s_abort);
          ok = false;
          break;
        }
        tc_fence_after();
        store_operand<F16>(tmem + lb + 384 + 64 * hf, reinterpret_cast<const float*>(dp));
        store_operand<F16>(tmem + lb + 384 + 64 * hf + 32, reinterpret_cast<const float*>(dp + 32));
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar_addr(c.ds_full));
      }
      if (!ok) break;
      if (!wait_warp(bar_addr(c.done), ii & 1)) {
        fail(&s_abort);
        ok = false;
        break;
      }
      ++ii;
      tc_fence_after();
#pragma unroll
      for (int cq = 0; cq < D / 64; ++cq) {
        const int col = hf * (D / 2) + cq * 32;  // dQ columns of this half
        uint32_t o[32];
        tmem_ld32(tmem + lb + 256 + col, o);
        if (in && a.dq_mode != 0) {  // fp32 dQ: a stored value is p + 0, like a first addition
          float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.dq) +
                                                  ((int64_t)t * a.H + itm.h) * D + col);
          float4 prev[8];  // all loads in flight before the first add
#pragma unroll
          for (int q = 0; q < 8; ++q)
            prev[q] = a.dq_mode == 2 ? dst[q] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float4 v;
            v.x = __fadd_rn(prev[q].x, __uint_as_float(o[q * 4 + 0]) * a.scale);
            v.y = __fadd_rn(prev[q].y, __uint_as_float(o[q * 4 + 1]) * a.scale);
            v.z = __fadd_rn(prev[q].z, __uint_as_float(o[q * 4 + 2]) * a.scale);
            v.w = __fadd_rn(prev[q].w, __uint_as_float(o[q * 4 + 3]) * a.scale);
            dst[q] = v;
          }
        } else if (in) {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<bf16*>(a.dq) +
                                                ((int64_t)t * a.H + itm.h) * D + col);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(o[q * 8 + 0]) * a.scale, __uint_as_float(o[q * 8 + 1]) * a.scale);
            v.y = pack_bf16(__uint_as_float(o[q * 8 + 2]) * a.scale, __uint_as_float(o[q * 8 + 3]) * a.scale);
            v.z = pack_bf16(__uint_as_float(o[q * 8 + 4]) * a.scale, __uint_as_float(o[q * 8 + 5]) * a.scale);
            v.w = pack_bf16(__uint_as_float(o[q * 8 + 6]) * a.scale, __uint_as_float(o[q * 8 + 7]) * a.scale);
            dst[q] = v;
          }
        }
      }
      // dQ's TMEM columns are rewritten (accumulate = 0) only by the next
      // item's first dQ product, which waits for this warp's next ds_full
      tc_fence_before();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

// ===========================================================================
// dK / dV
// ===========================================================================
constexpr int kStg = 2;  // Q/dO stages of attn_dkdv_tc
// attn_dkdv_tc runs 16 warps: 0-7 compute, 8-11 epilogue, 12 TMA producer,
// 13 TMEM allocator + MMA issuer, 14-15 idle.  Registers per thread after the
// split: compute 168, epilogue 96, the rest 80 (block total 65,536, the
// 512 x 128 it is launched with).
constexpr int kKvThr = 512;
constexpr int kKvEpi0 = 8, kKvProducer = 12, kKvMma = 13;
constexpr int kKvLaunchRegs = 128;
constexpr uint32_t kRegsCompute = 168, kRegsEpi = 96, kRegsRest = 80;
static_assert(8 * 32 * kRegsCompute + 4 * 32 * kRegsEpi + 4 * 32 * kRegsRest <=
                  kKvThr * kKvLaunchRegs, "register split exceeds the launch allocation");
constexpr int kEpiThreads = 128;

template <int D>
struct KvLayout {
  static constexpr int TILE = (D / 64) * kBox;
  static constexpr int K = 0;
  static constexpr int V = TILE;
  static constexpr int Q = 2 * TILE;
  static constexpr int DO = Q + kStg * TILE;
  static constexpr int BYTES = DO + kStg * TILE;
};

struct __align__(16) QInfo {  // per-query data of one 128-query step
  int lo[128];
  int hi[128];
  float nlse2[128];  // -LSE * log2(e)
  float dl[128];
  int max_lo, min_hi;
  int pad[2];
};

struct KvCtl {
  QInfo qinfo[kStg];
  uint64_t k_full, k_free, v_full, v_free;  // single K and V tiles of the item
  uint64_t q_full[kStg], qi_full[kStg], q_empty[kStg];
  uint64_t s_full, dp_full, p_full, ds_full, done, mma_done;
  uint64_t dv_free, dk_free;  // the epilogue warps have read the item's dV / dK out of TMEM
  uint32_t tmem;
  int abort;
};
// per-warp staging of the dK / dV epilogue follows KvCtl (16-byte aligned)
__host__ __device__ constexpr int kv_ctl_bytes() { return (int)((sizeof(KvCtl) + 15) & ~(size_t)15); }
constexpr int kStageBytes = 4 * 32 * 32 * 4;  // 4 epilogue warps x 32 rows x 32 fp32
// the staging buffers start on a 1024-byte boundary: the 128-byte swizzle of
// the bulk copies is a function of the shared-memory address
template <int D>
__host__ __device__ constexpr int kv_stage_offset() {
  return (KvLayout<D>::BYTES + kv_ctl_bytes() + 1023) & ~1023;
}


// Per query step i the MMA thread issues S^T_i, then the previous step's
// dK_{i-1} (once dS^T_{i-1} is in TMEM), then dP^T_i, then dV_i (once P^T_i
// is in TMEM).  While the compute warps turn S^T_i into P^T_i the tensor core
// runs dK_{i-1} and dP^T_i; while they form dS^T_i it runs dV_i and S^T_{i+1}.
// dP^T_i is committed only after the MMA thread has consumed ds_full(i-1) and
// S^T_{i+1} only after it has consumed p_full(i), so no per-step barrier gets
// two phases ahead of its waiter.
template <int D, bool F16>
__global__ void __launch_bounds__(kKvThr, 1)
attn_dkdv_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
             const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
             const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
             const __grid_constant__ BwdArgs a) {
  using L = KvLayout<D>;
  constexpr int BOXES = D / 64;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // launched early after the work-order kernel: its order and totals must be
  // complete and visible before any item is read
  pdl_wait();
  const MetaView m = meta_view(a.meta);
  if (a.n_ranks > 1 ? !meta_ok_grouped(a) : !meta_ok_bwd(a, m.hdr)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sb = smem_u32(smem_raw);
  if (sb & 1023u) {
    if (threadIdx.x == 0) atomicCAS(&g_status_bwd_tc, 0, (int)CP_ERR_UNSUPPORTED);
    return;
  }
  KvCtl& c = *reinterpret_cast<KvCtl*>(smem_raw + L::BYTES);
  volatile int& s_abort = *reinterpret_cast<volatile int*>(&c.abort);
  // key blocks: of the T keys, or in ring mode of every shard (blocks per shard
  // times the shards)
  const int n_kb = a.ring ? a.ring_cp * (int)n_tiles_of(a.s_local) : (int)n_tiles_of(a.T);
  const int n_items = n_kb * a.H;

  if (threadIdx.x == 0) {
    c.abort = 0;
    mbar_init(bar_addr(c.k_full), 1);
    mbar_init(bar_addr(c.k_free), 1);
    mbar_init(bar_addr(c.v_full), 1);
    mbar_init(bar_addr(c.v_free), 1);
    for (int s = 0; s < kStg; ++s) {
      mbar_init(bar_addr(c.q_full[s]), 1);
      mbar_init(bar_addr(c.qi_full[s]), 32);
      mbar_init(bar_addr(c.q_empty[s]), 1);
    }
    mbar_init(bar_addr(c.s_full), 1);
    mbar_init(bar_addr(c.dp_full), 1);
    mbar_init(bar_addr(c.p_full), kCompute);
    mbar_init(bar_addr(c.ds_full), kCompute);
    mbar_init(bar_addr(c.done), 1);
    mbar_init(bar_addr(c.mma_done), 1);
    mbar_init(bar_addr(c.dv_free), kEpiThreads);
    mbar_init(bar_addr(c.dk_free), kEpiThreads);
    fence_barrier_init();
  }
  if (warp == kKvMma) {
    tmem_alloc(smem_u32(&c.tmem), kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c.tmem;  // S^T [0,128) dP^T [128,256) dK [256,256+D) dV [256+D,256+2D)
  // Each warpgroup changes its register budget first thing in its own branch
  // (all four warps of a warpgroup execute the same setmaxnreg).
  if (warp >= kKvProducer) {
    reg_dealloc<kRegsRest>();
    if (warp == kKvProducer) {
    // all 32 lanes: lane 0 issues TMA, every lane loads per-query data
    int ii = 0, gs = 0, nk = 0, nv = 0;  // items, Q/dO steps, K and V tiles issued
    bool ok = true;
    auto wait_all = [&](uint32_t b, uint32_t parity) -> bool {
      const bool w = mbar_wait(b, parity, &s_abort, kLimitNs);
      return __all_sync(0xffffffffu, w);
    };
    for (int j = 0; ok && j * (int)gridDim.x < n_items; ++j) {
      const int k = snake_item(j, blockIdx.x, gridDim.x);
      if (k >= n_items) continue;
      const Item it = kv_item(a, m, k, n_kb);
      if (it.nb == 0) continue;
      const int j0 = (a.ring ? it.shard * a.s_local : 0) + it.tile * 128;  // first key row
      // single K (V) tile: free once the previous item's last S^T (dP^T) retired
      if (!wait_all(bar_addr(c.k_free), (ii & 1) ^ 1)) {
        if (lane == 0) fail(&s_abort);
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(bar_addr(c.k_full), L::TILE);
#pragma unroll
        for (int b = 0; b < BOXES; ++b)
          tma_load_3d(sb + L::K + b * kBox, &tm_k, bar_addr(c.k_full), b * 64, it.h, j0);
      }
      ++nk;
      if (!wait_all(bar_addr(c.v_free), (ii & 1) ^ 1)) {
        if (lane == 0) fail(&s_abort);
        ok = false;
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(bar_addr(c.v_full), L::TILE);
#pragma unroll
        for (int b = 0; b < BOXES; ++b)
          tma_load_3d(sb + L::V + b * kBox, &tm_v, bar_addr(c.v_full), b * 64, it.h, j0);
      }
      ++nv;
      ++ii;
      // the item's query tiles: one rank's block list, or every rank's in
      // rank order (rank r's rows at r * s_local of the concatenated Q / dO)
      const bool grouped = a.n_ranks > 1;
      for (int r = 0; ok && r < (grouped ? a.n_ranks : 1); ++r) {
        const int32_t* row_lo = m.row_lo;
        const int32_t* row_hi = m.row_hi;
        const int2* list = it.list;
        if (grouped) {
          const void* src = kv_source(a, it.shard, r);
          if (!src) continue;  // (ring mode) rank r never holds this shard
          const MetaView mr = meta_view(src);
          row_lo = mr.row_lo;
          row_hi = mr.row_hi;
          list = mr.klists + (kListBytes / 8) * it.tile;
        }
        const int nb = grouped ? list[0].y : it.nb;
        const int row0 = grouped ? r * a.s_local : 0;
        const int64_t ro = grouped ? (int64_t)r * a.H * a.s_local : 0;  // lse / delta of rank r
        Iter bi;
        bi.init(list + 1, min(list[0].x, kListCap));
        for (int i = 0; i < nb; ++i, bi.next(), ++gs) {
          const int st = gs % kStg;
          if (!wait_all(bar_addr(c.q_empty[st]), ((gs / kStg) & 1) ^ 1)) {
            if (lane == 0) fail(&s_abort);
            ok = false;
            break;
          }
          const int q0 = bi.b * 128;
          if (lane == 0) {
            mbar_arrive_expect_tx(bar_addr(c.q_full[st]), 2 * L::TILE);
#pragma unroll
            for (int b = 0; b < BOXES; ++b) {
              tma_load_3d(sb + L::Q + st * L::TILE + b * kBox, &tm_q, bar_addr(c.q_full[st]),
                          b * 64, it.h, row0 + q0);
              tma_load_3d(sb + L::DO + st * L::TILE + b * kBox, &tm_do, bar_addr(c.q_full[st]),
                          b * 64, it.h, row0 + q0);
            }
          }
          QInfo& qi = c.qinfo[st];
          int mlo = INT_MIN, mhi = INT_MAX;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int cq = lane + 32 * e;
            const int t = q0 + cq;
            const bool in = t < a.s_local;
            const int hi = in ? row_hi[t] : -1;
            const int lo = in ? row_lo[t] : 0;
            qi.lo[cq] = lo;
            qi.hi[cq] = hi;
            qi.nlse2[cq] = hi >= 0 ? -a.lse[ro + (int64_t)it.h * a.s_local + t] * kLog2ef : 0.f;
            qi.dl[cq] = hi >= 0 ? a.delta[ro + (int64_t)it.h * a.s_local + t] : 0.f;
            mlo = max(mlo, lo);
            mhi = min(mhi, hi);
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            mlo = max(mlo, __shfl_xor_sync(0xffffffffu, mlo, o));
            mhi = min(mhi, __shfl_xor_sync(0xffffffffu, mhi, o));
          }
          if (lane == 0) {
            qi.max_lo = mlo;
            qi.min_hi = mhi;
          }
          __syncwarp();
          mbar_arrive(bar_addr(c.qi_full[st]));
        }
      }
    }
    if (lane == 0) {
      // drain: every copy this CTA issued must land before shared memory goes away
      int never = 0;
      if (nk > 0) mbar_wait(bar_addr(c.k_full), (nk - 1) & 1, &never, kLimitNs);
      if (nv > 0) mbar_wait(bar_addr(c.v_full), (nv - 1) & 1, &never, kLimitNs);
      for (int i = max(0, gs - kStg); i < gs; ++i)
        mbar_wait(bar_addr(c.q_full[i % kStg]), (i / kStg) & 1, &never, kLimitNs);
    }
  } else if (warp == kKvMma) {
    // The whole warp runs the issue loop (uniform control flow, warp-uniform
    // waits); one elected lane issues each MMA and commit.
    auto wait_w = [&](uint32_t b, uint32_t parity) -> bool {
      const bool w = mbar_wait(b, parity, &s_abort, kLimitNs);
      return __all_sync(0xffffffffu, w);
    };
    {
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false, F16);
      constexpr uint32_t idG = idesc_bf16_f32(128, D, false, true, F16);
      // operand descriptors at the tiles' first bytes (K-major, and Q / dO as MN-major)
      const uint64_t dsc_k = sdesc_sw128(sb + L::K, 16, 1024);
      const uint64_t dsc_v = sdesc_sw128(sb + L::V, 16, 1024);
      const uint64_t dsc_q = sdesc_sw128(sb + L::Q, 16, 1024);
      const uint64_t dsc_do = sdesc_sw128(sb + L::DO, 16, 1024);
      const uint64_t dsc_qmn = sdesc_sw128(sb + L::Q, kBox, 1024);
      const uint64_t dsc_domn = sdesc_sw128(sb + L::DO, kBox, 1024);
      int ii = 0, gs = 0;
      int pend = -1, pend_st = 0, pend_item = 0;  // step whose dK product is still to be issued
      bool pend_first = false;
      // dK += dS^T Q : A = dS^T (TMEM over dP^T), B = Q tile as MN-major.  An
      // item's first dK starts dK afresh: the epilogue warps must have read the
      // previous item's dK out of TMEM first.
      auto issue_dk = [&]() -> bool {
        if (!wait_w(bar_addr(c.ds_full), pend & 1)) return false;
        if (pend_first && pend_item > 0 &&
            !wait_w(bar_addr(c.dk_free), (pend_item - 1) & 1))
          return false;
        tc_fence_after();
        const uint64_t bq = sdesc_add(dsc_qmn, pend_st * L::TILE);
        // dS^T is the sum of two bf16 terms: two products per k-step
#pragma unroll (D == 128 && !F16 ? 4 : 8)  // (spill-free in the 80-register share)
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t b = sdesc_add(bq, kk * 2048);
          umma_bf16_ts_w(tmem + 256, tmem + 128 + hilo_col(kk), b, idG,
                       (!pend_first || kk > 0) ? 1u : 0u);
          if (!F16) umma_bf16_ts_w(tmem + 256, tmem + 128 + hilo_col(kk) + 16, b, idG, 1u);
        }
        umma_commit_w(bar_addr(c.q_empty[pend_st]));
        return true;
      };
      bool ok = true;
      for (int j = 0; ok && j * (int)gridDim.x < n_items; ++j) {
        const int k = snake_item(j, blockIdx.x, gridDim.x);
        if (k >= n_items) continue;
        Item it;  // (only its step count matters here)
        it.nb = kv_item_nb(a, m, k, n_kb);
        if (it.nb == 0) continue;
        const int cur = ii++;
        if (!wait_w(bar_addr(c.k_full), cur & 1)) {
          fail(&s_abort);
          break;
        }
        for (int i = 0; i < it.nb; ++i, ++gs) {
          const int st = gs % kStg;
          if (!wait_w(bar_addr(c.q_full[st]), (gs / kStg) & 1)) {
            fail(&s_abort);
            ok = false;
            break;
          }
          // S^T_gs overwrites P^T_{gs-1}: its reader dV_{gs-1} was issued
          // earlier by this thread, and p_full(gs-1) (waited before it) means
          // the compute warps are done with S^T_{gs-1}
          tc_fence_after();
          const uint64_t bq = sdesc_add(dsc_q, st * L::TILE);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = kmajor_off(kk);
            umma_bf16_w(tmem, sdesc_add(dsc_k, off), sdesc_add(bq, off), idS, kk > 0);
          }
          umma_commit_w(bar_addr(c.s_full));
          if (i == it.nb - 1) umma_commit_w(bar_addr(c.k_free));
          // dK of the previous step; its ds_full also means the compute warps
          // have read dP^T_{gs-1}, which dP^T_gs overwrites
          if (pend >= 0 && !issue_dk()) {
            fail(&s_abort);
            ok = false;
            break;
          }
          if (i == 0 && !wait_w(bar_addr(c.v_full), cur & 1)) {
            fail(&s_abort);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bd = sdesc_add(dsc_do, st * L::TILE);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = kmajor_off(kk);
            umma_bf16_w(tmem + 128, sdesc_add(dsc_v, off), sdesc_add(bd, off), idS, kk > 0);
          }
          umma_commit_w(bar_addr(c.dp_full));
          if (i == it.nb - 1) umma_commit_w(bar_addr(c.v_free));
          if (!wait_w(bar_addr(c.p_full), gs & 1) ||
              (i == 0 && cur > 0 &&
               !wait_w(bar_addr(c.dv_free), (cur - 1) & 1))) {
            fail(&s_abort);
            ok = false;
            break;
          }
          tc_fence_after();
          // dV += P^T dO : A = P^T (TMEM over S^T), B = dO tile as MN-major (N = d);
          // an item's first dV starts afresh once the previous dV has been read out.
          // P^T is the sum of two bf16 terms (rounded P, then its remainder), so
          // the product carries P to about 16 bits instead of bf16's 8.
          const uint64_t bdm = sdesc_add(dsc_domn, st * L::TILE);
#pragma unroll (D == 128 && !F16 ? 4 : 8)  // (spill-free in the 80-register share)
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t b = sdesc_add(bdm, kk * 2048);
            umma_bf16_ts_w(tmem + 256 + D, tmem + ts_col(kk), b, idG, (i > 0 || kk > 0) ? 1u : 0u);
            if (!F16) umma_bf16_ts_w(tmem + 256 + D, tmem + ts_col(kk) + 32, b, idG, 1u);
          }
          pend = gs;
          pend_st = st;
          pend_first = (i == 0);
          pend_item = cur;
        }
        if (!ok) break;
        if (!issue_dk()) {
          fail(&s_abort);
          break;
        }
        pend = -1;
        umma_commit_w(bar_addr(c.done));
      }
      umma_commit_w(bar_addr(c.mma_done));
      int never = 0;
      mbar_wait(bar_addr(c.mma_done), 0, &never, kLimitNs);
    }
    }
  } else if (warp >= kKvEpi0) {
    // ------------------------------------------------------------ epilogue warps 8-11
    reg_dealloc<kRegsEpi>();
    // Warp w reads TMEM lanes 32*(w%4).. (one key row per lane) of the finished
    // item's dV, then dK, 32 columns at a time, releases each accumulator as
    // soon as its last columns are in registers, and adds them into the fp32
    // accumulators.  This item is the only writer of these rows in this launch:
    // one fp32 add per element, done in L2 without a round trip.  Each 32 x 32
    // chunk goes into a private shared-memory buffer in the 128-byte swizzle
    // order (16-byte unit u of row r at u ^ (r & 7), conflict-free) and one
    // bulk tensor copy per chunk adds it to (or, first rank, stores it in) the
    // accumulators: cp.reduce.async.bulk.tensor ... .add, issued by lane 0.
    const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;
    float* stg = reinterpret_cast<float*>(smem_raw + kv_stage_offset<D>()) +
                 (warp - kKvEpi0) * 32 * 32;
    const uint32_t stg_s = smem_u32(stg);
    auto wait_warp = [&](uint32_t b, uint32_t parity) -> bool {
      const bool w = mbar_wait(b, parity, &s_abort, kLimitNs);
      return __all_sync(0xffffffffu, w);
    };
    int ii = 0;
    for (int j = 0; j * (int)gridDim.x < n_items; ++j) {
      const int k = snake_item(j, blockIdx.x, gridDim.x);
      if (k >= n_items) continue;
      const Item itm = kv_item(a, m, k, n_kb);
      if (itm.nb == 0) {
        // no query of this rank attends these keys: a stored partial is zero
        if (a.rs) {
          const int kr = (a.ring ? itm.shard * a.s_local : 0) + itm.tile * 128 + (warp & 3) * 32 +
                         lane;
          const int64_t t = rs_dst_row(a, kr, a.ring ? (itm.shard + 1) * a.s_local : a.T);
          if (t >= 0) {
            uint4* dk = reinterpret_cast<uint4*>(a.dk16 + (t * a.H + itm.h) * D);
            uint4* dv = reinterpret_cast<uint4*>(a.dv16 + (t * a.H + itm.h) * D);
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 4
            for (int u = 0; u < D / 8; ++u) {
              dk[u] = z;
              dv[u] = z;
            }
          }
        } else if (a.store) {
          const int rb = (a.ring ? itm.shard * a.s_local : 0) + itm.tile * 128 + (warp & 3) * 32;
          const int row_end = a.ring ? (itm.shard + 1) * a.s_local : a.T;
          const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32)
#pragma unroll
            for (int it = 0; it < 8; ++it) {
              const int kr = rb + (lane >> 3) + 4 * it;
              if (kr < row_end) {
                const int64_t o = ((int64_t)kr * a.H + itm.h) * D + c0 + 4 * (lane & 7);
                *reinterpret_cast<float4*>(a.dk + o) = z;
                *reinterpret_cast<float4*>(a.dv + o) = z;
              }
            }
        }
        continue;
      }
      if (!wait_warp(bar_addr(c.done), ii & 1)) {
        fail(&s_abort);
        break;
      }
      ++ii;
      tc_fence_after();
      // first key row of this warp, and the end of the key rows the item owns
      // (ring mode: its shard's; the 32-row chunks never straddle a shard end,
      // s_local being a multiple of 32 there)
      const int rbase = (a.ring ? itm.shard * a.s_local : 0) + itm.tile * 128 + (warp & 3) * 32;
      const int row_end = a.ring ? (itm.shard + 1) * a.s_local : a.T;
      // fused scatter: this lane's key row and its destination row (-1: none)
      const int64_t drow = a.rs ? rs_dst_row(a, rbase + lane, row_end) : -1;
#pragma unroll 1
      for (int ch = 0; ch < 2 * (D / 32); ++ch) {
        const bool is_v = ch < D / 32;  // dV first, then dK
        const int c0 = (is_v ? ch : ch - D / 32) * 32;
        uint32_t v[32];
        tmem_ld32(tmem + lb + 256 + (is_v ? D : 0) + c0, v);
        if (ch == D / 32 - 1 || ch == 2 * (D / 32) - 1) {
          tc_fence_before();
          mbar_arrive(bar_addr(is_v ? c.dv_free : c.dk_free));
        }
        const float sc = is_v ? 1.f : a.scale;
        if (a.rs) {
          // the lane's 32 values of its row, rounded to bf16 as the stored
          // fp32 sum would be (+0 first), straight to the destination row
          if (drow >= 0) {
            uint4* d = reinterpret_cast<uint4*>((is_v ? a.dv16 : a.dk16) +
                                                (drow * a.H + itm.h) * D + c0);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w[e] = pack_bf16(__fadd_rn(__uint_as_float(v[8 * u + 2 * e]) * sc, 0.f),
                                 __fadd_rn(__uint_as_float(v[8 * u + 2 * e + 1]) * sc, 0.f));
              d[u] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
          continue;
        }
        // the previous chunk's bulk copy has finished reading the staging buffer
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
        // row `lane` of the 32 x 32 chunk, its 16-byte units in the 128-byte
        // swizzle order the tensor map's box uses (unit u at u ^ (row & 7));
        // a stored partial is p + 0, the value the first addition into a
        // cleared buffer gives
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          float4 x = make_float4(__uint_as_float(v[4 * u]) * sc, __uint_as_float(v[4 * u + 1]) * sc,
                                 __uint_as_float(v[4 * u + 2]) * sc,
                                 __uint_as_float(v[4 * u + 3]) * sc);
          if (a.store)
            x = make_float4(__fadd_rn(x.x, 0.f), __fadd_rn(x.y, 0.f), __fadd_rn(x.z, 0.f),
                            __fadd_rn(x.w, 0.f));
          *reinterpret_cast<float4*>(stg + lane * 32 + ((u ^ (lane & 7)) * 4)) = x;
        }
        fence_proxy_async_smem();
        __syncwarp();
        // one bulk copy moves the chunk: rows rbase.. (those past T are not
        // written), columns c0.., added in L2 (or stored by the first rank)
        if (lane == 0 && rbase < row_end) {  // (a box wholly past the item's rows is skipped)
          const CUtensorMap* map = is_v ? &tm_dv : &tm_dk;
          if (a.store) tma_store_3d(map, stg_s, c0, itm.h, rbase);
          else tma_reduce_add_3d(map, stg_s, c0, itm.h, rbase);
          bulk_commit();
        }
      }
    }
    // every bulk copy of this warp has landed before the CTA (and its shared
    // memory) goes away
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  } else {
    reg_alloc<kRegsCompute>();
    const int row = (warp & 3) * 32 + lane;  // TMEM lane = key row of the block
    const int hf = warp >> 2;                // column half: queries [64hf, 64hf+64)
    const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;
    const float sl2 = a.scale_log2;
    auto wait_warp = [&](uint32_t b, uint32_t parity) -> bool {
      const bool w = mbar_wait(b, parity, &s_abort, kLimitNs);
      return __all_sync(0xffffffffu, w);
    };
    int gs = 0;
    bool ok = true;
    for (int j = 0; ok && j * (int)gridDim.x < n_items; ++j) {
      const int k = snake_item(j, blockIdx.x, gridDim.x);
      if (k >= n_items) continue;
      const Item itm = kv_item(a, m, k, n_kb);
      if (itm.nb == 0) continue;  // no query of this rank attends these keys
      const int key = itm.tile * 128 + row;
      for (int i = 0; i < itm.nb; ++i, ++gs) {
        const int st = gs % kStg;
        if (!wait_warp(bar_addr(c.s_full), gs & 1) ||
            !wait_warp(bar_addr(c.qi_full[st]), (gs / kStg) & 1)) {
          fail(&s_abort);
          ok = false;
          break;
        }
        tc_fence_after();
        const QInfo& qi = c.qinfo[st];
        const float* nl = qi.nlse2 + 64 * hf;
        const float* dl = qi.dl + 64 * hf;
        float p[64];
        tmem_ld32(tmem + lb + 64 * hf, reinterpret_cast<uint32_t*>(p));
        tmem_ld32(tmem + lb + 64 * hf + 32, reinterpret_cast<uint32_t*>(p + 32));
        // (scalar arithmetic here: the paired forms need register pairs that this
        // kernel's compute warps cannot spare without spilling)
        const float4* l4 = reinterpret_cast<const float4*>(nl);
        if (key >= qi.max_lo && key <= qi.min_hi) {  // every query of the step sees this key
#pragma unroll
          for (int c4 = 0; c4 < 16; ++c4) {
            const float4 l = l4[c4];
            p[4 * c4 + 0] = ex2_approx(fmaf(p[4 * c4 + 0], sl2, l.x));
            p[4 * c4 + 1] = ex2_approx(fmaf(p[4 * c4 + 1], sl2, l.y));
            p[4 * c4 + 2] = ex2_approx(fmaf(p[4 * c4 + 2], sl2, l.z));
            p[4 * c4 + 3] = ex2_approx(fmaf(p[4 * c4 + 3], sl2, l.w));
          }
        } else {
          const int4* lo4 = reinterpret_cast<const int4*>(qi.lo + 64 * hf);
          const int4* hi4 = reinterpret_cast<const int4*>(qi.hi + 64 * hf);
#pragma unroll
          for (int c4 = 0; c4 < 16; ++c4) {
            const float4 l = l4[c4];
            const int4 lo = lo4[c4], hi = hi4[c4];
            p[4 * c4 + 0] = (key >= lo.x && key <= hi.x) ? ex2_approx(fmaf(p[4 * c4 + 0], sl2, l.x)) : 0.f;
            p[4 * c4 + 1] = (key >= lo.y && key <= hi.y) ? ex2_approx(fmaf(p[4 * c4 + 1], sl2, l.y)) : 0.f;
            p[4 * c4 + 2] = (key >= lo.z && key <= hi.z) ? ex2_approx(fmaf(p[4 * c4 + 2], sl2, l.z)) : 0.f;
            p[4 * c4 + 3] = (key >= lo.w && key <= hi.w) ? ex2_approx(fmaf(p[4 * c4 + 3], sl2, l.w)) : 0.f;
          }
        }
        {  // P^T -> TMEM as two bf16 terms over this half's S^T columns: the
           // rounded P (first 32 columns) and its rounding remainder (next 32)
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            if (F16) {
              uint32_t ph[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) ph[e] = pack_f16(p[32 * cc + 2 * e], p[32 * cc + 2 * e + 1]);
              tmem_st16(tmem + lb + 64 * hf + 16 * cc, ph);
            } else {
              uint32_t ph[16], pl[16];
              split_bf16(p + 32 * cc, ph, pl);
              tmem_st16(tmem + lb + 64 * hf + 16 * cc, ph);
              tmem_st16(tmem + lb + 64 * hf + 32 + 16 * cc, pl);
            }
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar_addr(c.p_full));
        if (!wait_warp(bar_addr(c.dp_full), gs & 1)) {
          fail(&s_abort);
          ok = false;
          break;
        }
        tc_fence_after();
        // dS^T = P^T (dP^T - Delta) over the dP^T columns just read, as hi and
        // lo bf16 terms
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t dp[32];
          const uint32_t col = tmem + lb + 128 + 64 * hf + 32 * cc;
          tmem_ld32(col, dp);
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 d = reinterpret_cast<const float4*>(dl)[cc * 8 + e4];
            const int c0 = cc * 32 + 4 * e4;
            dp[4 * e4] = __float_as_uint(p[c0] * (__uint_as_float(dp[4 * e4]) - d.x));
            dp[4 * e4 + 1] = __float_as_uint(p[c0 + 1] * (__uint_as_float(dp[4 * e4 + 1]) - d.y));
            dp[4 * e4 + 2] = __float_as_uint(p[c0 + 2] * (__uint_as_float(dp[4 * e4 + 2]) - d.z));
            dp[4 * e4 + 3] = __float_as_uint(p[c0 + 3] * (__uint_as_float(dp[4 * e4 + 3]) - d.w));
          }
          store_operand<F16>(col, reinterpret_cast<const float*>(dp));
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar_addr(c.ds_full));
      }
      if (!ok) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kKvMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

// Heaviest-first work orders of the grouped and ring launches, ranked by
// comparison against every entry (stable for equal counts).  One block; tot
// holds n ints of scratch.
//   family 1 (dK/dV, rank-grouped or ring): the key blocks (ring mode: of every
//     shard, entry shard * blocks-per-shard + block) with their query-tile
//     count summed over the sources (the ranks, or the ranks' steps that hold
//     the shard);
//   family 0 (dQ, ring mode): the rank's query tiles with their key-block count
//     summed over its ring steps.
// Metadata that does not match (the attention kernel then writes nothing)
// gives the identity order and its lists are not read.
constexpr int kOrdThreads = 1024, kOrdChunk = 4096;
__global__ void __launch_bounds__(kOrdThreads, 1)
grouped_korder_kernel(const BwdArgs a, int family, int n, int* tot, int2* order) {
  __shared__ int s_t[kOrdChunk];
  __shared__ int s_ok;
  if (threadIdx.x == 0)
    s_ok = (family == 0 ? meta_ok_steps(a) : meta_ok_grouped(a)) ? 1 : 0;
  __syncthreads();
  if (!s_ok) {
    for (int q = threadIdx.x; q < n; q += blockDim.x) order[q] = make_int2(q, 0);
    return;
  }
  const int per = (int)n_tiles_of(a.s_local);  // key blocks per shard (ring mode)
  for (int q = threadIdx.x; q < n; q += blockDim.x) {
    int t = 0;
    if (family == 0) {
      for (int i = 0; i < a.n_steps; ++i)
        t += meta_view(step_meta(a, i)).qlists[(kListBytes / 8) * q].y;
    } else {
      const int shard = a.ring ? q / per : 0, kb = a.ring ? q % per : q;
      for (int r = 0; r < a.n_ranks; ++r) {
        const void* src = kv_source(a, shard, r);
        if (src) t += meta_view(src).klists[(kListBytes / 8) * kb].y;
      }
    }
    tot[q] = t;
  }
  __syncthreads();
  for (int q0 = 0; q0 < n; q0 += blockDim.x) {
    const int q = q0 + threadIdx.x;
    const int mine = q < n ? tot[q] : 0;
    int rank = 0;
    for (int c0 = 0; c0 < n; c0 += kOrdChunk) {
      const int cn = min(kOrdChunk, n - c0);
      __syncthreads();
      for (int i = threadIdx.x; i < cn; i += blockDim.x) s_t[i] = tot[c0 + i];
      __syncthreads();
      if (q < n)
        for (int i = 0; i < cn; ++i) {
          const int o = s_t[i];
          rank += (o > mine || (o == mine && c0 + i < q)) ? 1 : 0;
        }
    }
    if (q < n) order[rank] = make_int2(q, mine);
  }
}

// One launch, with programmatic stream serialization when pdl is set (the
// kernel may then start before the previous grid in the stream has finished).
template <typename... P, typename... A>
cudaError_t launch_ex(void (*kernel)(P...), int grid, int block, int smem, cudaStream_t s,
                      bool pdl, A&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<A&&>(args)...);
}

// parts: 1 = the dQ kernel, 2 = the dK/dV kernel (rank-grouped when
// a.n_ranks > 1: Q / dO maps over the n_ranks * s_local concatenated rows).
// pdl bit 1: the dQ kernel may start while the previous grid finishes (it
// reads nothing that grid writes); bit 2: so may the dK/dV work-order kernel,
// and the dK/dV kernel may start as the order kernel completes (it waits for
// the order before reading it).
template <int D, bool F16>
int launch_bwd_tc(const void* q, const void* k, const void* v, const void* dout,
                  const BwdArgs& a, int parts, cudaStream_t s, int kv_rows_arg = 0, int pdl = 0) {
  alignas(64) CUtensorMap mq, mdo, mk, mv, mdk{}, mdv{};
  int st;
  const int q_rows = a.s_local * (a.n_ranks > 1 ? a.n_ranks : 1);
  if ((st = tma::make_thd_map(&mq, q, q_rows, a.H, D, 128, F16)) != CP_OK) return st;
  if ((st = tma::make_thd_map(&mdo, dout, q_rows, a.H, D, 128, F16)) != CP_OK) return st;
  const int kv_rows = kv_rows_arg > 0 ? kv_rows_arg : a.T;  // rows of K, V, dK, dV
  if ((st = tma::make_thd_map(&mk, k, kv_rows, a.H, D, 128, F16)) != CP_OK) return st;
  if ((st = tma::make_thd_map(&mv, v, kv_rows, a.H, D, 128, F16)) != CP_OK) return st;
  if ((parts & 2) && !a.rs) {  // (the dQ pass and the fused scatter use no fp32 map)
    if ((st = tma::make_f32_rows_map(&mdk, a.dk, kv_rows, a.H, D)) != CP_OK) return st;
    if ((st = tma::make_f32_rows_map(&mdv, a.dv, kv_rows, a.H, D)) != CP_OK) return st;
  }
  const int dq_smem = DqLayout<D>::BYTES + (int)sizeof(DqCtl);
  const int kv_smem = kv_stage_offset<D>() + kStageBytes;
  if (cudaFuncSetAttribute(attn_dq_tc<D, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           dq_smem) != cudaSuccess ||
      cudaFuncSetAttribute(attn_dkdv_tc<D, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kv_smem) != cudaSuccess)
    return CP_ERR_CUDA;
  const int sms = cpthd_host::sm_count();
  if (parts & 1) {
    if (a.n_steps > 1) {  // ring mode: the rank's query tiles by their count over the steps
      grouped_korder_kernel<<<1, kOrdThreads, 0, s>>>(a, 0, (int)n_tiles_of(a.s_local),
                                                      a.gorder_tot, const_cast<int2*>(a.gorder));
      if ((st = cpthd_host::launch_status()) != CP_OK) return st;
    }
    const int64_t q_items = n_tiles_of(a.s_local) * (int64_t)a.H;
    if (launch_ex(attn_dq_tc<D, F16>, (int)(q_items < sms ? q_items : sms), kThr, dq_smem, s,
                  (pdl & 1) != 0, mq, mdo, mk, mv, a) != cudaSuccess)
      return CP_ERR_CUDA;
    if ((st = cpthd_host::launch_status()) != CP_OK) return st;
  }
  if (!(parts & 2)) return CP_OK;
  // key blocks: of the T keys, or in ring mode of every shard
  const int n_kb = a.ring ? a.ring_cp * (int)n_tiles_of(a.s_local) : (int)n_tiles_of(a.T);
  if (a.n_ranks > 1) {
    if (launch_ex(grouped_korder_kernel, 1, kOrdThreads, 0, s, (pdl & 2) != 0, a, 1, n_kb,
                  a.gorder_tot, const_cast<int2*>(a.gorder)) != cudaSuccess)
      return CP_ERR_CUDA;
    if ((st = cpthd_host::launch_status()) != CP_OK) return st;
  }
  const int64_t k_items = (int64_t)n_kb * a.H;
  // the register split inside attn_dkdv_tc assumes exactly kKvLaunchRegs per thread at launch
  static int kv_regs = -1;
  if (kv_regs < 0) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, attn_dkdv_tc<D, F16>) != cudaSuccess) return CP_ERR_CUDA;
    kv_regs = fa.numRegs;
  }
  if (kv_regs != kKvLaunchRegs) return CP_ERR_UNSUPPORTED;
  if (launch_ex(attn_dkdv_tc<D, F16>, (int)(k_items < sms ? k_items : sms), kKvThr, kv_smem, s,
                (pdl & 2) != 0, mq, mdo, mk, mv, mdk, mdv, a) != cudaSuccess)
    return CP_ERR_CUDA;
  return cpthd_host::launch_status();
}

}  // namespace
}  // namespace cpthd

// Internal entry used by the backward entry points (arguments validated, Delta
// already computed into `delta`).
int cpthd_attn_bwd_tc(const void* q, const void* k, const void* v, const void* dout,
                      const float* lse, const float* delta, void* dq, float* dk, float* dv,
                      const void* meta, size_t meta_bytes, int T, int H, int D, int s_local,
                      int cp, int rank, int strategy, float scale, float scale_log2,
                      int mode, int f16, cudaStream_t s, int pdl) {
  using namespace cpthd;
  BwdArgs a{};
  a.lse = lse;
  a.delta = delta;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.meta = meta;
  a.meta_bytes = meta_bytes;
  a.T = T; a.H = H; a.s_local = s_local; a.cp = cp; a.rank = rank; a.strategy = strategy;
  a.scale = scale;
  a.scale_log2 = scale_log2;
  a.store = mode & 1;
  a.dq_mode = (mode & 2) ? 1 : (mode & 4) ? 2 : 0;
  a.n_ranks = 1;
  const int parts = (mode & kBwdDqOnly) ? 1 : 3;
  if (f16)
    return D == 64 ? launch_bwd_tc<64, true>(q, k, v, dout, a, parts, s, 0, pdl)
                   : launch_bwd_tc<128, true>(q, k, v, dout, a, parts, s, 0, pdl);
  return D == 64 ? launch_bwd_tc<64, false>(q, k, v, dout, a, parts, s, 0, pdl)
                 : launch_bwd_tc<128, false>(q, k, v, dout, a, parts, s, 0, pdl);
}

// Internal entry of the rank-grouped dK/dV: one launch over every key block,
// each walking the attending query tiles of all cp ranks, stored once into the
// fp32 dK / dV (every row written), or with dk16 / dv16 given, rounded to bf16
// into row rs_row[j] (j without an index) of the rank-concatenated outputs
// (the reduce-scatter's scatter fused in; dk / dv unused).  q_all / dout_all
// are the rank-concatenated [cp * s_local, H, D] operands, lse_all / delta_all
// [cp][H][s_local], meta_all the cp ranks' metadata meta_stride bytes apart;
// scratch holds n_kb ints and then (16-aligned) n_kb int2 of the work order.
int cpthd_attn_dkdv_grouped_tc(const void* q_all, const void* k, const void* v,
                               const void* dout_all, const float* lse_all,
                               const float* delta_all, float* dk, float* dv,
                               const void* meta_all, size_t meta_stride, int T, int H, int D,
                               int s_local, int cp, int strategy, float scale, float scale_log2,
                               int f16, void* scratch, cudaStream_t s, void* dk16, void* dv16,
                               const int32_t* rs_row, int pdl) {
  using namespace cpthd;
  BwdArgs a{};
  a.lse = lse_all;
  a.delta = delta_all;
  a.dk = dk;
  a.dv = dv;
  a.rs = dk16 != nullptr;
  a.rs_row = rs_row;
  a.dk16 = reinterpret_cast<uint16_t*>(dk16);
  a.dv16 = reinterpret_cast<uint16_t*>(dv16);
  a.meta = meta_all;
  a.meta_bytes = meta_stride;
  a.T = T; a.H = H; a.s_local = s_local; a.cp = cp; a.rank = 0; a.strategy = strategy;
  a.scale = scale;
  a.scale_log2 = scale_log2;
  a.store = 1;
  a.n_ranks = cp;
  a.meta_stride = (int64_t)meta_stride;
  a.gorder_tot = reinterpret_cast<int*>(scratch);
  a.gorder = reinterpret_cast<const int2*>(reinterpret_cast<char*>(scratch) +
                                           grouped_order_offset(T));
  if (f16)
    return D == 64 ? launch_bwd_tc<64, true>(q_all, k, v, dout_all, a, 2, s, 0, pdl)
                   : launch_bwd_tc<128, true>(q_all, k, v, dout_all, a, 2, s, 0, pdl);
  return D == 64 ? launch_bwd_tc<64, false>(q_all, k, v, dout_all, a, 2, s, 0, pdl)
                 : launch_bwd_tc<128, false>(q_all, k, v, dout_all, a, 2, s, 0, pdl);
}

// Internal entry of the ring backward in one pass (arguments validated, every
// rank's Delta in delta_all): per rank one dQ launch over all its ring steps
// (dQ stored once, bf16), then one dK/dV launch over the key blocks of every
// shard, each walking the ranks that hold the shard at some step, stored once
// (fp32, rank-concatenated rows).  ring_meta: rank r's step metadata at
// r * rank_stride, step i at + i * step_bytes (cp_size = 1 blocks); q_all /
// dout_all / dq_all / k_shards / v_shards / dk / dv are [cp * s_local, H, D];
// lse_all / delta_all [cp][H][s_local]; scratch: ring_bwd_scratch_bytes.  With
// dk16 / dv16 given, dK / dV go out rounded to bf16 there instead (dk / dv
// unused): the cast of the reduce-scatter in the same epilogue.
int cpthd_attn_bwd_ring_tc(const void* q_all, const void* k_shards, const void* v_shards,
                           const void* dout_all, const float* lse_all, const float* delta_all,
                           void* dq_all, float* dk, float* dv, const void* ring_meta,
                           size_t step_bytes, size_t rank_stride, int H, int D, int s_local,
                           int cp, int strategy, float scale, float scale_log2, int f16,
                           void* scratch, cudaStream_t s, void* dk16, void* dv16) {
  using namespace cpthd;
  const int n_qt = (int)n_tiles_of(s_local);
  int* tot = reinterpret_cast<int*>(scratch);
  int2* order = reinterpret_cast<int2*>(reinterpret_cast<char*>(scratch) +
                                        ring_bwd_order_offset(s_local, cp));
  const int kv_rows = s_local * cp;  // the ranks' shards side by side
  auto launch = [&](const void* q, const void* dout, const BwdArgs& a, int parts) {
    if (f16)
      return D == 64 ? launch_bwd_tc<64, true>(q, k_shards, v_shards, dout, a, parts, s, kv_rows)
                     : launch_bwd_tc<128, true>(q, k_shards, v_shards, dout, a, parts, s, kv_rows);
    return D == 64 ? launch_bwd_tc<64, false>(q, k_shards, v_shards, dout, a, parts, s, kv_rows)
                   : launch_bwd_tc<128, false>(q, k_shards, v_shards, dout, a, parts, s, kv_rows);
  };
  const size_t row_bytes = (size_t)H * D * 2;
  for (int r = 0; r < cp; ++r) {  // dQ of rank r over its ring steps
    BwdArgs a{};
    a.lse = lse_all + (size_t)r * H * s_local;
    a.delta = delta_all + (size_t)r * H * s_local;
    a.dq = reinterpret_cast<char*>(dq_all) + (size_t)r * s_local * row_bytes;
    a.meta = reinterpret_cast<const char*>(ring_meta) + rank_stride * r;
    a.meta_bytes = step_bytes;
    a.T = s_local; a.H = H; a.s_local = s_local; a.cp = 1; a.rank = 0; a.strategy = strategy;
    a.scale = scale;
    a.scale_log2 = scale_log2;
    a.dq_mode = 0;
    a.n_ranks = 1;
    a.n_steps = strategy == (int)CP_NO_LOAD_BALANCE ? r + 1 : cp;
    a.step_stride = (int64_t)step_bytes;
    a.ring_rank = r;
    a.ring_cp = cp;
    a.gorder = order;
    a.gorder_tot = tot;
    if (n_qt == 0) continue;
    const int st = launch(reinterpret_cast<const char*>(q_all) + (size_t)r * s_local * row_bytes,
                          reinterpret_cast<const char*>(dout_all) + (size_t)r * s_local * row_bytes,
                          a, 1);
    if (st != CP_OK) return st;
  }
  BwdArgs a{};  // dK / dV of every shard
  a.lse = lse_all;
  a.delta = delta_all;
  a.dk = dk;
  a.dv = dv;
  a.rs = dk16 != nullptr;  // bf16 straight out: the shards are already rank-concatenated
  a.dk16 = reinterpret_cast<uint16_t*>(dk16);
  a.dv16 = reinterpret_cast<uint16_t*>(dv16);
  a.meta = ring_meta;
  a.meta_bytes = step_bytes;
  a.T = s_local; a.H = H; a.s_local = s_local; a.cp = 1; a.rank = 0; a.strategy = strategy;
  a.scale = scale;
  a.scale_log2 = scale_log2;
  a.store = 1;
  a.ring = 1;
  a.n_ranks = cp;
  a.ring_cp = cp;
  a.step_stride = (int64_t)step_bytes;
  a.meta_stride = (int64_t)rank_stride;
  a.gorder = order;
  a.gorder_tot = tot;
  return launch(q_all, dout_all, a, 2);
}

extern "C" int cpthd_status_bwd_tc(int reset) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, cpthd::g_status_bwd_tc, sizeof(int)) != cudaSuccess)
    return CP_ERR_CUDA;
  if (reset) {
    int z = 0;
    if (cudaMemcpyToSymbol(cpthd::g_status_bwd_tc, &z, sizeof(int)) != cudaSuccess)
      return CP_ERR_CUDA;
  }
  return v;
}
