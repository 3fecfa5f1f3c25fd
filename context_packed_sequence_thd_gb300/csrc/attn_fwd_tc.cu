// attn_fwd_tc.cu -- causal varlen attention forward of one CP rank on the
// Blackwell tensor cores (tcgen05 + TMEM + TMA), built for sm_103a.
//
// The tensor-core operands (Q, K, V and the probabilities P) are all bf16 or
// all fp16 (F16), accumulation fp32.
//
// What it computes ("[PyTorch] Add no-load-balance THD all-gather CP", §Why
// and §Scope and constraints): for every local query row t of the rank (global
// row g of document i), O_t = softmax_j(scale * q_t . k_j) v_j over the keys
// j in [cup[i], g], and LSE_t in natural log; padding rows get O = 0,
// LSE = -inf.  Both DUAL_CHUNK_SWAP chunks of a rank go through one launch:
// the key range of every row comes from the rank's row tables.
//
// Persistent kernel: one CTA per SM walks a static list of work items
// (128-row query tile, head), heaviest tiles first, dealt to the CTAs in
// rounds of alternating direction.  The pipeline never drains between items: all barrier phases
// follow global counters, Q is double buffered, and an item's epilogue is
// deferred until the next item's first block has been handed to the tensor
// core, so it overlaps the next item's S products.  10 warps:
//   warps 0-7  softmax: TMEM lane r = query row r, shared by warps r/32 and
//              r/32+4 which take one half of the key columns each.  Loads S
//              from TMEM, masks by the row's key range, online softmax in the
//              log2 domain over its own key half -- its own running max and
//              sum, and its own accumulator O_half, so the two warps of a row
//              never wait for each other within an item -- rescales O_half
//              only when its max grows by more than 2^8, writes P (bf16
//              pairs) back into TMEM over S (before any O rescale, so S and O
//              are never live in registers together).  The epilogue combines
//              the halves (maxima and sums swapped once through shared
//              memory), normalises and stores O / LSE, and frees O_0 / O_1.
//   warp 8     TMA producer: Q per item into one of two buffers, K tiles into
//              a 3-stage ring released as soon as S is done, V tiles into a
//              2-stage ring released after P V; K runs one block ahead of V.
//              With a query index (cp_attn_fwd_gather) the Q tile is read
//              straight from the unsharded source, every lane gathering four
//              rows per copy (tile::gather4).
//   warp 9     TMEM allocator and MMA issuer (one elected lane per MMA):
//              S[g%2] = Q K_g^T (M=128, N=128, K=D, both operands K-major in
//              shared memory) and O_h += P_g[:, keys of half h] V_g[keys of
//              half h] (M=128, N=D, K=64 each; A = P from TMEM, B = V as an
//              MN-major shared operand); an item's first P V waits until the
//              previous item's epilogue has read O_0 / O_1.  TMEM: S0 cols
//              [0,128), S1 [128,256), O_0 [256,256+D), O_1 [256+D,256+2D).
// The MMA of S_{g+1} overlaps the softmax of S_g; P_g goes to the other S
// buffer than P_{g-1}, and the softmax waits for P V_{g-1} only when it has to
// rescale O, so consecutive P V products are issued back to back.
// Key blocks per tile come from the precomputed block lists (document and
// causal skipping), in increasing order.
// Every wait is bounded (mbar_wait): a wait that runs out sets the device
// status word to CP_ERR_TIMEOUT, the CTA drains its own copies / MMAs and
// frees its TMEM before it returns.
#include <math.h>

#include "common.cuh"
#include "sm100.cuh"
#include "tma_host.cuh"

namespace cpthd {

static __device__ int g_status_fwd_tc;

namespace {

using namespace sm100;
using bf16 = __nv_bfloat16;

constexpr int TBM = 128;           // query rows per tile
constexpr int TBN = 128;           // keys per block
constexpr int kThreadsTc = 320;    // 10 warps
constexpr int kSoftmax = 256;      // threads of the softmax warps 0-7
constexpr int kProdWarp = 8, kMmaWarp = 9;
constexpr int kKStages = 3;        // K ring depth (released after S)
constexpr int kVStages = 2;        // V ring depth (released after P V)
constexpr int kBoxBytes = 128 * 128;  // one 128-row x 128-byte TMA box
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 4000000000ull;  // default bound of a wait
constexpr float kLn2f = 0.6931471805599453f;

template <int D>
struct Layout {
  static constexpr int BOXES = D / 64;            // 64-element boxes along D
  static constexpr int TILE = BOXES * kBoxBytes;  // one Q / K / V tile
  static constexpr int Q = 0;                     // two Q buffers
  static constexpr int K = Q + 2 * TILE;
  static constexpr int V = K + kKStages * TILE;
  static constexpr int BYTES = V + kVStages * TILE;
};

template <int D>
__host__ __device__ constexpr uint32_t o_col(int b) { return 256 + b * D; }

struct TcArgs {
  bf16* o;
  bf16* o_resid;  // nullable: O - bf16(O), rounded to bf16 (the backward's Delta reads O + it)
  float* lse;
  const int32_t* q_idx;  // nullable: query row t is row q_idx[t] of a q_rows-row source
  int q_rows;
  const void* meta;
  size_t meta_bytes;
  int T, H, s_local, cp, rank, strategy;
  float scale_log2;
  uint64_t limit_ns;  // bound of every mbarrier wait
  int skip_first_k;   // failure-detection test only: CTA 0 never loads its first K tile
  // ring mode (n_steps > 1): every ring step of rank ring_rank in one pass.
  // meta is step 0's metadata (cp_size = 1, as cp_p2p_index writes it) and
  // step i's lies step_stride bytes further per step; step i's keys are the
  // shard of rank (ring_rank - i) mod ring_cp, rows shard_rows * that rank of
  // the K / V tensors (kv_rows rows in all); rorder holds the rank's query
  // tiles heaviest first by their block count summed over the steps.
  int n_steps;
  int64_t step_stride;
  int ring_rank, ring_cp, shard_rows, kv_rows;
  const int2* rorder;
};

// Metadata of ring step i (step 0 outside ring mode).
__device__ __forceinline__ const void* step_meta(const TcArgs& a, int i) {
  return reinterpret_cast<const char*>(a.meta) + a.step_stride * i;
}

struct Bars {
  uint64_t q_full[2];
  uint64_t q_free[2];  // all S products of the item using Q buffer b are done
  uint64_t k_full[kKStages];
  uint64_t k_empty[kKStages];
  uint64_t v_full[kVStages];
  uint64_t v_empty[kVStages];
  uint64_t s_full[2];
  uint64_t p_full[2];   // P_g ready: p_full[g % 2]
  uint64_t o_ready[2];  // P V_g done: o_ready[g % 2]
  uint64_t o_free;      // the item's epilogue has read O_0 / O_1 (one phase per item)
  uint64_t mma_done;
};
// Why two alternating barriers suffice for s_full / p_full / o_ready: the MMA
// thread issues S_g after P V_{g-2}, so when the softmax holds S_g every
// P V up to g-2 is complete, and P V_{g+1} cannot be issued before the
// softmax has produced P_{g+1}.  A parity wait on o_ready[(g-1) % 2] (or, for
// a deferred epilogue at block L+1, on o_ready[L % 2]) therefore always sees
// exactly the phase it is waiting for.  o_free completes one phase per item
// epilogue; the MMA thread waits for item q-1's before item q's first P V,
// and item q's epilogue needs that P V done, so it is never two phases behind.

// Barriers and small per-CTA state, placed right after the tiles in the
// dynamic shared memory (the kernel has no static shared memory, so the
// dynamic window starts 1024-aligned and the tiles need no alignment slack).
struct Ctl {
  Bars bars;
  uint64_t pair[4][2];  // epilogue exchange of running max / sum of softmax warps w, w+4
  uint32_t tmem;
  int abort;
  int pad[2];
  float red[2][2][TBM];  // [exchange parity][column half][row]
};

__device__ __forceinline__ bool meta_ok_tc(const TcArgs& a, const MetaHeader* h) {
  bool ok = true;
  int bad = 0;
  for (int i = 0; i < a.n_steps && ok; ++i) {  // every ring step's metadata in ring mode
    const MetaHeader* hi = i == 0 ? h : reinterpret_cast<const MetaHeader*>(step_meta(a, i));
    ok = meta_matches(hi, a.meta_bytes, a.T, a.s_local, a.cp, a.rank, a.strategy);
    if (!ok) bad = hi->status != 0 ? hi->status : (int)CP_ERR_METADATA;
  }
  if (!ok && threadIdx.x == 0) atomicCAS(&g_status_fwd_tc, 0, bad);
  return ok;
}

// Ring mode: the rank's query tiles heaviest first by their block count summed
// over the ring steps (each step's tile list header), ranked by comparison
// against every tile (stable for equal counts).  One block; tot holds n_qt
// ints of scratch.  Metadata that does not match leaves the identity order
// with zero counts (the attention kernel then writes nothing).
constexpr int kOrdThreads = 1024, kOrdChunk = 4096;
__global__ void __launch_bounds__(kOrdThreads, 1)
ring_order_kernel(const TcArgs a, int* tot, int2* order) {
  __shared__ int s_t[kOrdChunk];
  __shared__ int s_ok;
  const int n = (int)n_tiles_of(a.s_local);
  if (threadIdx.x == 0) {
    int ok = 1;
    for (int i = 0; i < a.n_steps && ok; ++i)
      ok = meta_matches(reinterpret_cast<const MetaHeader*>(step_meta(a, i)), a.meta_bytes, a.T,
                        a.s_local, a.cp, a.rank, a.strategy) ? 1 : 0;
    s_ok = ok;
  }
  __syncthreads();
  if (!s_ok) {
    for (int q = threadIdx.x; q < n; q += blockDim.x) order[q] = make_int2(q, 0);
    return;
  }
  for (int q = threadIdx.x; q < n; q += blockDim.x) {
    int t = 0;
    for (int i = 0; i < a.n_steps; ++i) t += meta_view(step_meta(a, i)).qlists[(kListBytes / 8) * q].y;
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

__device__ __forceinline__ void fail(volatile int* abort) {
  *abort = 1;
  atomicCAS(&g_status_fwd_tc, 0, (int)CP_ERR_TIMEOUT);
}

// One work item: its tile, head and number of key blocks (ring mode: summed
// over the ring steps).
struct Item {
  int tile, t0, h, nb;
  // item k: the q-th heaviest tile of head h, heaviest first over all heads
  __device__ void load(const TcArgs& a, const MetaView& m, int k, int n_qt) {
    int q;
    item_of(k, n_qt, a.H, a.H, &q, &h);
    const int2 o = (a.n_steps > 1 ? a.rorder : m.qorder)[min(max(q, 0), n_qt - 1)];
    tile = min(max(o.x, 0), n_qt - 1);
    t0 = tile * TBM;
    nb = o.y;
  }
};

struct Iter {  // flattened walk over an item's key-block intervals
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

// The key blocks of a work item in order: the tile's block list, or in ring
// mode the lists of the rank's ring steps one after another (the steps with
// blocks), each step's blocks in its shard.  Producer and softmax warps walk
// the same sequence; b is a block of the current step's shard, kv_off the
// shard's first row in the K / V tensors.
struct Walk {
  const TcArgs* a;
  Iter bi;
  int tile, step, left, kv_off;
  __device__ void init(const TcArgs& args, int t) {
    a = &args;
    tile = t;
    step = -1;
    left = 0;
    kv_off = 0;
    advance();
  }
  __device__ void advance() {
    while (left == 0 && step + 1 < a->n_steps) {
      ++step;
      const int2* list = meta_view(step_meta(*a, step)).qlists + (kListBytes / 8) * tile;
      left = list[0].y;
      bi.init(list + 1, min(list[0].x, kListCap));
      kv_off = a->ring_cp > 0
                   ? ((a->ring_rank - step + a->ring_cp) % a->ring_cp) * a->shard_rows
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

template <int D, bool F16>
__global__ void __launch_bounds__(kThreadsTc, 1)
attn_fwd_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_v, const TcArgs a) {
  using L = Layout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const MetaView m = meta_view(a.meta);
  if (!meta_ok_tc(a, m.hdr)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sb = smem_u32(smem_raw);  // tiles need 1024-byte alignment (128B swizzle)
  if (sb & 1023u) {
    if (threadIdx.x == 0) atomicCAS(&g_status_fwd_tc, 0, (int)CP_ERR_UNSUPPORTED);
    return;
  }
  Ctl& ctl = *reinterpret_cast<Ctl*>(smem_raw + L::BYTES);
  Bars& bars = ctl.bars;
  volatile int& s_abort = *reinterpret_cast<volatile int*>(&ctl.abort);
  const int n_qt = (int)n_tiles_of(a.s_local);
  const int n_items = n_qt * a.H;

  auto bar = [](uint64_t& b) { return smem_u32(&b); };
  if (threadIdx.x == 0) {
    ctl.abort = 0;
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(bars.q_full[b]), 1);
      mbar_init(bar(bars.q_free[b]), 1);
      mbar_init(bar(bars.s_full[b]), 1);
      mbar_init(bar(bars.p_full[b]), kSoftmax);
      mbar_init(bar(bars.o_ready[b]), 1);
    }
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(bar(bars.k_full[s]), 1);
      mbar_init(bar(bars.k_empty[s]), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(bar(bars.v_full[s]), 1);
      mbar_init(bar(bars.v_empty[s]), 1);
    }
    mbar_init(bar(bars.o_free), kSoftmax);
    mbar_init(bar(bars.mma_done), 1);
    for (int w = 0; w < 4; ++w) {
      mbar_init(bar(ctl.pair[w][0]), 64);
      mbar_init(bar(ctl.pair[w][1]), 64);
    }
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&ctl.tmem), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem;

  if (warp == kProdWarp) {
    // ---------------------------------------------------------------- TMA producer
    // The whole warp walks the items; lane 0 waits, arms the barriers and
    // issues the tiled copies, and every lane takes part in the row gathers
    // of a fused-gather Q tile (four rows per lane).
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    // lane 0 waits; the result is the warp's
    auto wait0 = [&](uint64_t& b, uint32_t parity) -> bool {
      const bool w = lane == 0 ? mbar_wait(bar(b), parity, &s_abort, a.limit_ns) : true;
      return __shfl_sync(0xffffffffu, w, 0);
    };
    int ii = 0, g = 0, v_issued = 0;
    int pv_h = 0, pv_key = 0;  // V of block v_issued still to load (when v_issued < g)
    bool ok = true;
    auto load_v = [&]() -> bool {
      const int vs = v_issued % kVStages;
      if (!wait0(bars.v_empty[vs], ((v_issued / kVStages) & 1) ^ 1)) return false;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(bars.v_full[vs]), L::TILE);
#pragma unroll
        for (int b = 0; b < L::BOXES; ++b)
          tma_load_3d(sb + L::V + vs * L::TILE + b * kBoxBytes, &tm_v, bar(bars.v_full[vs]),
                      b * 64, pv_h, pv_key);
      }
      ++v_issued;
      return true;
    };
    for (int j = 0; ok && j * (int)gridDim.x < n_items; ++j) {
      const int k = snake_item(j, blockIdx.x, gridDim.x);
      if (k >= n_items) continue;
      Item it;
      it.load(a, m, k, n_qt);
      if (it.nb == 0) continue;
      const int qb = ii & 1;
      if (!wait0(bars.q_free[qb], ((ii >> 1) & 1) ^ 1)) {
        if (lane == 0) fail(&s_abort);
        break;
      }
      if (lane == 0) mbar_arrive_expect_tx(bar(bars.q_full[qb]), L::TILE);
      if (a.q_idx) {
        // fused partition gather: the tile's rows come straight from the
        // source by the rank's index, lane l gathering rows 4l..4l+3 (rows
        // past s_local repeat the last row; they are masked)
        __syncwarp();
        const int t = it.t0 + 4 * lane, last = a.s_local - 1;
        int r[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) r[e] = __ldg(a.q_idx + min(t + e, last));
        bool bad = false;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if ((unsigned)r[e] >= (unsigned)a.q_rows) {  // outside the source: report, read row 0
            bad = true;
            r[e] = 0;
          }
        }
        if (bad) atomicCAS(&g_status_fwd_tc, 0, (int)CP_ERR_INVALID_ARG);
#pragma unroll
        for (int b = 0; b < L::BOXES; ++b)
          tma_gather4_2d(sb + L::Q + qb * L::TILE + b * kBoxBytes + lane * 512, &tm_q,
                         bar(bars.q_full[qb]), it.h * D + b * 64, r[0], r[1], r[2], r[3]);
      } else if (lane == 0) {
#pragma unroll
        for (int b = 0; b < L::BOXES; ++b)
          tma_load_3d(sb + L::Q + qb * L::TILE + b * kBoxBytes, &tm_q, bar(bars.q_full[qb]),
                      b * 64, it.h, it.t0);
      }
      ++ii;
      Walk w;
      w.init(a, it.tile);
      for (int j = 0; j < it.nb; ++j, w.next()) {
        const int ks = g % kKStages;
        if (!wait0(bars.k_empty[ks], ((g / kKStages) & 1) ^ 1)) {
          if (lane == 0) fail(&s_abort);
          ok = false;
          break;
        }
        const int key0 = w.kv_off + w.b() * TBN;  // the block's first row in K / V
        // (the failure-detection test leaves CTA 0's first K tile unloaded: the
        // MMA thread's bounded wait for it runs out and the CTA drains)
        if (lane == 0 && !(a.skip_first_k && blockIdx.x == 0 && g == 0)) {
          mbar_arrive_expect_tx(bar(bars.k_full[ks]), L::TILE);
#pragma unroll
          for (int b = 0; b < L::BOXES; ++b)
            tma_load_3d(sb + L::K + ks * L::TILE + b * kBoxBytes, &tm_k, bar(bars.k_full[ks]),
                        b * 64, it.h, key0);
        }
        ++g;
        if (v_issued < g - 1 && !load_v()) {  // V lags K by one block
          if (lane == 0) fail(&s_abort);
          ok = false;
          break;
        }
        pv_h = it.h;
        pv_key = key0;
      }
    }
    if (ok && v_issued < g && !load_v() && lane == 0) fail(&s_abort);
    // drain: every copy this CTA issued must land before shared memory goes away
    if (lane == 0) {
      int never = 0;
      for (int i = max(0, ii - 2); i < ii; ++i)
        mbar_wait(bar(bars.q_full[i & 1]), (i >> 1) & 1, &never, a.limit_ns);
      for (int j = max(0, g - kKStages); j < g; ++j)
        mbar_wait(bar(bars.k_full[j % kKStages]), (j / kKStages) & 1, &never, a.limit_ns);
      for (int j = max(0, v_issued - kVStages); j < v_issued; ++j)
        mbar_wait(bar(bars.v_full[j % kVStages]), (j / kVStages) & 1, &never, a.limit_ns);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    // The whole warp runs the issue loop (uniform control flow, warp-uniform
    // waits); one elected lane issues each MMA and commit.
    auto wait_w = [&](uint32_t b, uint32_t parity) -> bool {
      const bool w = mbar_wait(b, parity, &s_abort, a.limit_ns);
      return __all_sync(0xffffffffu, w);
    };
    {
      constexpr uint32_t idS = idesc_bf16_f32(128, TBN, false, false, F16);
      constexpr uint32_t idO = idesc_bf16_f32(128, D, false, true, F16);
      // operand descriptors at the tiles' first bytes, built once (an MMA's
      // descriptor is then one 64-bit add): Q and K K-major, V MN-major
      const uint64_t dsc_q = sdesc_sw128(sb + L::Q, 16, 1024);
      const uint64_t dsc_k = sdesc_sw128(sb + L::K, 16, 1024);
      const uint64_t dsc_v = sdesc_sw128(sb + L::V, kBoxBytes, 1024);
      // the previous block's P V is issued after the next block's S
      int pv_g = -1, pv_item = 0;  // pv_item: the CTA's non-empty items begun before pv_g's
      bool pv_first = false;
      auto issue_pv = [&]() -> bool {
        const int vs = pv_g % kVStages;
        if (!wait_w(bar(bars.p_full[pv_g & 1]), (pv_g >> 1) & 1) ||
            !wait_w(bar(bars.v_full[vs]), (pv_g / kVStages) & 1))
          return false;
        // an item's first P V starts O_0 / O_1 afresh: the previous item's
        // epilogue must have read them
        if (pv_first && pv_item > 0 && !wait_w(bar(bars.o_free), (pv_item - 1) & 1)) return false;
        tc_fence_after();
        // A = P from TMEM: keys [0,64) over columns [0,32) and keys [64,128)
        // over [64,96) of S_g's buffer (written by the two column halves);
        // each key half accumulates into its own O (O_0, O_1), against its
        // own running max
        const uint64_t bv = sdesc_add(dsc_v, vs * L::TILE);
        const uint32_t aP = tmem + (pv_g & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < TBN / 16; ++kk)
          umma_bf16_ts_w(tmem + o_col<D>(kk >> 2), aP + (kk >> 2) * 64 + (kk & 3) * 8,
                         sdesc_add(bv, kk * 2048), idO, (!pv_first || (kk & 3) > 0) ? 1u : 0u);
        umma_commit_w(bar(bars.v_empty[vs]));
        umma_commit_w(bar(bars.o_ready[pv_g & 1]));
        return true;
      };
      int ii = 0, g = 0;
      bool ok = true;
      for (int j = 0; ok && j * (int)gridDim.x < n_items; ++j) {
        const int k = snake_item(j, blockIdx.x, gridDim.x);
        if (k >= n_items) continue;
        Item it;
        it.load(a, m, k, n_qt);
        if (it.nb == 0) continue;
        const int qb = ii & 1;
        if (!wait_w(bar(bars.q_full[qb]), (ii >> 1) & 1)) {
          fail(&s_abort);
          break;
        }
        ++ii;
        for (int j = 0; j < it.nb; ++j, ++g) {
          const int ks = g % kKStages, buf = g & 1;
          // S_g overwrites P_{g-2} (same TMEM columns); P V_{g-2} was issued
          // earlier by this warp and the MMAs of one issuer run in order
          if (!wait_w(bar(bars.k_full[ks]), (g / kKStages) & 1)) {
            fail(&s_abort);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bq = sdesc_add(dsc_q, qb * L::TILE), bk = sdesc_add(dsc_k, ks * L::TILE);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
            umma_bf16_w(tmem + buf * 128, sdesc_add(bq, off), sdesc_add(bk, off), idS,
                        kk > 0 ? 1u : 0u);
          }
          umma_commit_w(bar(bars.s_full[buf]));
          umma_commit_w(bar(bars.k_empty[ks]));
          if (j == it.nb - 1) umma_commit_w(bar(bars.q_free[qb]));
          if (pv_g >= 0 && !issue_pv()) {
            fail(&s_abort);
            ok = false;
            break;
          }
          pv_g = g;
          pv_first = (j == 0);
          if (pv_first) pv_item = ii - 1;
        }
      }
      if (ok && pv_g >= 0 && !issue_pv()) fail(&s_abort);
      // drain: all MMAs issued by this warp must finish before TMEM is freed
      umma_commit_w(bar(bars.mma_done));
      int never = 0;
      mbar_wait(bar(bars.mma_done), 0, &never, a.limit_ns);
    }
  } else {
    // ---------------------------------------------------------------- softmax (warps 0-7)
    // Warps w and w+4 share TMEM lanes 32*(w%4).. (one query row per lane):
    // warp w takes key columns [0,64) of each block, warp w+4 columns
    // [64,128).  Each half runs its own online softmax over its key columns
    // -- its own running max, row sum and accumulator O_hf (the P V products
    // of its keys) -- so the two warps never wait for each other within an
    // item.  The epilogue combines the halves once per item: with M the
    // larger of the two running maxima, O = sum_h O_h 2^(m_h - M) /
    // sum_h l_h 2^(m_h - M) (maxima and sums swapped through shared memory),
    // each warp normalising and storing one half of the D columns.
    const int row = (warp & 3) * 32 + lane;  // = TMEM lane
    const int hf = warp >> 2;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const float sl2 = a.scale_log2;
    // waits of the softmax warps are made warp-uniform (tcgen05.ld/st are
    // .sync.aligned): the warp proceeds only when every lane saw the phase
    auto wait_warp = [&](uint32_t b, uint32_t parity) -> bool {
      const bool w = mbar_wait(b, parity, &s_abort, a.limit_ns);
      return __all_sync(0xffffffffu, w);
    };
    // exchange u of the two warps of a pair: publish a value, wait for the
    // partner's (bounded, like every other wait), return the partner's value
    int u = 0;
    auto exchange = [&](float v, float* out) -> bool {
      ctl.red[u & 1][hf][row] = v;
      mbar_arrive(bar(ctl.pair[warp & 3][u & 1]));
      const bool w = wait_warp(bar(ctl.pair[warp & 3][u & 1]), (u >> 1) & 1);
      if (w) *out = ctl.red[u & 1][hf ^ 1][row];
      ++u;
      return w;
    };
    // the CTA's next non-empty work item after round j (n_items if none)
    auto next_item = [&](int j) -> int {
      for (++j; j * (int)gridDim.x < n_items; ++j) {
        const int k = snake_item(j, blockIdx.x, gridDim.x);
        if (k >= n_items) continue;
        Item nx;
        nx.load(a, m, k, n_qt);
        if (nx.nb > 0) return k;
      }
      return n_items;
    };
    // the finished item whose O still has to be normalised and stored
    struct Pending {
      int t, h, last;
      float m, l;
    } pend{0, 0, -1, 0.f, 0.f};
    auto epilogue = [&]() -> bool {
      if (!wait_warp(bar(bars.o_ready[pend.last & 1]), (pend.last >> 1) & 1)) return false;
      float m_other = 0.f, l_other = 0.f;
      if (!exchange(pend.m, &m_other) || !exchange(pend.l, &l_other)) return false;
      // the halves' weights against the larger running max (a half that saw
      // no key of the row has m = -inf, l = 0 and weight 0)
      const float m_max = fmaxf(pend.m, m_other);
      const float w_own = pend.m == -INFINITY ? 0.f : ex2_approx((pend.m - m_max) * sl2);
      const float w_oth = m_other == -INFINITY ? 0.f : ex2_approx((m_other - m_max) * sl2);
      const float l_tot = pend.l * w_own + l_other * w_oth;
      const float w0 = hf == 0 ? w_own : w_oth, w1 = hf == 0 ? w_oth : w_own;
      const bool in = pend.t < a.s_local;
      tc_fence_after();
      const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
      const float s0 = w0 * inv, s1 = w1 * inv;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        const int col = hf * (D / 2) + c * 32;
        uint32_t o[32], o1[32];
        tmem_ld32(tmem + lane_base + o_col<D>(0) + col, o);
        tmem_ld32(tmem + lane_base + o_col<D>(1) + col, o1);
        if (in) {
          const int64_t off = ((int64_t)pend.t * a.H + pend.h) * D + col;
          uint4* dst = reinterpret_cast<uint4*>(a.o + off);
          uint4* dst_r = reinterpret_cast<uint4*>(a.o_resid + off);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              x[e] = __uint_as_float(o[q * 8 + e]) * s0 + __uint_as_float(o1[q * 8 + e]) * s1;
            uint4 v;
            v.x = pack_bf16(x[0], x[1]);
            v.y = pack_bf16(x[2], x[3]);
            v.z = pack_bf16(x[4], x[5]);
            v.w = pack_bf16(x[6], x[7]);
            dst[q] = v;
            if (a.o_resid) {
              uint4 r;
              r.x = pack_bf16(x[0] - bf16_lo_f(v.x), x[1] - bf16_hi_f(v.x));
              r.y = pack_bf16(x[2] - bf16_lo_f(v.y), x[3] - bf16_hi_f(v.y));
              r.z = pack_bf16(x[4] - bf16_lo_f(v.z), x[5] - bf16_hi_f(v.z));
              r.w = pack_bf16(x[6] - bf16_lo_f(v.w), x[7] - bf16_hi_f(v.w));
              dst_r[q] = r;
            }
          }
        }
      }
      if (in && hf == 0)
        a.lse[(int64_t)pend.h * a.s_local + pend.t] =
            l_tot > 0.f ? (m_max * sl2 + log2f(l_tot)) * kLn2f : -INFINITY;
      // O_0 / O_1 are read: the next item's first P V may overwrite them
      tc_fence_before();
      mbar_arrive(bar(bars.o_free));
      pend.last = -1;
      return true;
    };

    int ii = 0, g = 0;
    bool ok = true;
    // row tables of the next non-empty item are fetched one item ahead
    int k_pre = next_item(-1);
    int lo_pre = 0, hi_pre = -1;
    if (k_pre < n_items) {
      Item f;
      f.load(a, m, k_pre, n_qt);
      const int t = f.t0 + row;
      lo_pre = t < a.s_local ? m.row_lo[t] : 0;
      hi_pre = t < a.s_local ? m.row_hi[t] : -1;
    }
    for (int j = 0; ok && j * (int)gridDim.x < n_items; ++j) {
      const int k = snake_item(j, blockIdx.x, gridDim.x);
      if (k >= n_items) continue;
      Item itm;
      itm.load(a, m, k, n_qt);
      const int t = itm.t0 + row;
      if (itm.nb == 0) {  // no real query row in this tile: O = 0, LSE = -inf
        if (t < a.s_local) {
          const int64_t off = ((int64_t)t * a.H + itm.h) * D + hf * (D / 2);
          uint4* dst = reinterpret_cast<uint4*>(a.o + off);
#pragma unroll
          for (int c = 0; c < D / 16; ++c) dst[c] = make_uint4(0, 0, 0, 0);
          if (a.o_resid) {
            uint4* dst_r = reinterpret_cast<uint4*>(a.o_resid + off);
#pragma unroll
            for (int c = 0; c < D / 16; ++c) dst_r[c] = make_uint4(0, 0, 0, 0);
          }
          if (hf == 0) a.lse[(int64_t)itm.h * a.s_local + t] = -INFINITY;
        }
        continue;
      }
      int lo = lo_pre, hi = hi_pre;  // step 0's key range of the row (k == k_pre here)
      k_pre = next_item(j);
      if (k_pre < n_items) {
        Item f;
        f.load(a, m, k_pre, n_qt);
        const int tn = f.t0 + row;
        lo_pre = tn < a.s_local ? m.row_lo[tn] : 0;
        hi_pre = tn < a.s_local ? m.row_hi[tn] : -1;
      }
      ++ii;
      float m_run = -INFINITY, l_run = 0.f;  // this column half's running max and sum
      Walk w;
      w.init(a, itm.tile);
      int cur_step = 0;  // the ring step whose key range lo / hi hold
      for (int j = 0; j < itm.nb; ++j, w.next(), ++g) {
        const int buf = g & 1;
        if (w.step != cur_step) {  // ring mode: the row's key range in the next step's shard
          const MetaView ms = meta_view(step_meta(a, w.step));
          lo = t < a.s_local ? ms.row_lo[t] : 0;
          hi = t < a.s_local ? ms.row_hi[t] : -1;
          cur_step = w.step;
        }
        if (!wait_warp(bar(bars.s_full[buf]), (g >> 1) & 1)) {
          fail(&s_abort);
          ok = false;
          break;
        }
        tc_fence_after();
        float s[64];
        tmem_ld32(tmem + lane_base + buf * 128 + 64 * hf, reinterpret_cast<uint32_t*>(s));
        tmem_ld32(tmem + lane_base + buf * 128 + 64 * hf + 32,
                  reinterpret_cast<uint32_t*>(s + 32));

        const int k0 = w.b() * TBN + 64 * hf;  // key (of the step's shard) of this thread's first column
        if (!(lo <= k0 && hi >= k0 + 63)) {
          // column c is visible iff lo <= k0 + c <= hi: one unsigned compare of
          // c - (lo - k0) against hi - lo (a row with no key masks everything)
          const bool any = hi >= lo;
          const int c_lo = any ? lo - k0 : (1 << 30);
          const unsigned span = any ? (unsigned)(hi - lo) : 0u;
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if ((unsigned)(c - c_lo) > span) s[c] = -INFINITY;
        }
        // this half's row max: eight independent chains of three-input maxima
        float mx8[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          mx8[q] = fmax3(s[q], s[8 + q], s[16 + q]);
          mx8[q] = fmax3(mx8[q], s[24 + q], s[32 + q]);
          mx8[q] = fmax3(mx8[q], s[40 + q], s[48 + q]);
          mx8[q] = fmaxf(mx8[q], s[56 + q]);
        }
        const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                               fmaxf(mx8[6], mx8[7]));
        // The running max m_run is only moved (and O, l rescaled) when the new
        // block's max exceeds it by more than 8 in log2 units; otherwise the
        // stale max stays in use for this block's P, which then stays below
        // 2^8 -- P and l always use the same reference, so O/l is unchanged.
        // While m_run is still -inf every P so far was exactly 0, so O = 0 and
        // l = 0 need no rescale.
        float alpha = 1.f;
        if (m_run == -INFINITY || (mx - m_run) * sl2 > 8.f) {
          const float m_new = fmaxf(m_run, mx);
          if (m_run != -INFINITY) alpha = ex2_approx((m_run - m_new) * sl2);
          m_run = m_new;
        }
        const float mref = m_run == -INFINITY ? 0.f : m_run * sl2;
        // P = 2^(s * scale_log2 - mref): the scaling in paired FMAs, 2^x on
        // the SFU (with the two halves of a row no longer in lockstep, taking
        // a share on the FMA pipe by a polynomial measured 2-4% slower)
        const uint64_t scl2 = f2_pack(sl2, sl2), nref2 = f2_pack(-mref, -mref);
        uint64_t sum2[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) sum2[q] = f2_pack(0.f, 0.f);
#pragma unroll
        for (int c2 = 0; c2 < 32; ++c2) {
          float a, b;
          f2_unpack(f2_fma(f2_pack(s[2 * c2], s[2 * c2 + 1]), scl2, nref2), a, b);
          a = ex2_approx(a);
          b = ex2_approx(b);
          s[2 * c2] = a;
          s[2 * c2 + 1] = b;
          sum2[c2 & 3] = f2_add(sum2[c2 & 3], f2_pack(a, b));
        }
        float sum, sum_b;
        f2_unpack(f2_add(f2_add(sum2[0], sum2[1]), f2_add(sum2[2], sum2[3])), sum, sum_b);
        sum += sum_b;
        l_run = l_run * alpha + sum;

        {  // P (bf16 pairs) -> TMEM over the first 32 of this half's S columns;
           // written before any O rescale so that S is dead while O is in registers
          uint32_t pk[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) pk[e] = pack_op<F16>(s[2 * e], s[2 * e + 1]);
          tmem_st32(tmem + lane_base + buf * 128 + 64 * hf, pk);
        }
        // O only has to be complete (P V_{g-1} done) when it is rescaled; the
        // first block of an item starts a fresh accumulator.
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          const int pv = g - 1;
          if (!wait_warp(bar(bars.o_ready[pv & 1]), (pv >> 1) & 1)) {
            fail(&s_abort);
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {  // this half's accumulator, every column
            const uint32_t col = o_col<D>(hf) + c * 32;
            uint32_t o[32];
            tmem_ld32(tmem + lane_base + col, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tmem + lane_base + col, o);
          }
          tmem_st_wait();
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(bars.p_full[buf]));
        // the previous item's epilogue runs once this item's first block is
        // with the tensor core
        if (j == 0 && pend.last >= 0 && !epilogue()) {
          fail(&s_abort);
          ok = false;
          break;
        }
      }
      if (!ok) break;
      pend.t = t;
      pend.h = itm.h;
      pend.last = g - 1;
      pend.m = m_run;
      pend.l = l_run;
    }
    if (ok && pend.last >= 0 && !epilogue()) fail(&s_abort);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

template <int D, bool F16>
int launch_fwd_tc(const void* q, const void* k, const void* v, const TcArgs& a, cudaStream_t s) {
  alignas(64) CUtensorMap mq, mk, mv;
  int st;
  st = a.q_idx ? tma::make_row_gather_map(&mq, q, a.q_rows, a.H, D, F16)
               : tma::make_thd_map(&mq, q, a.s_local, a.H, D, 128, F16);
  if (st != CP_OK) return st;
  if ((st = tma::make_thd_map(&mk, k, a.kv_rows, a.H, D, 128, F16)) != CP_OK) return st;
  if ((st = tma::make_thd_map(&mv, v, a.kv_rows, a.H, D, 128, F16)) != CP_OK) return st;
  const int smem = Layout<D>::BYTES + (int)sizeof(Ctl);
  if (cudaFuncSetAttribute(attn_fwd_tc<D, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return CP_ERR_CUDA;
  const int64_t items = n_tiles_of(a.s_local) * (int64_t)a.H;
  const int grid = (int)(items < cpthd_host::sm_count() ? items : cpthd_host::sm_count());
  attn_fwd_tc<D, F16><<<grid, kThreadsTc, smem, s>>>(mq, mk, mv, a);
  return cpthd_host::launch_status();
}

}  // namespace
}  // namespace cpthd

// Internal entry used by cp_attn_fwd (arguments already validated).
int cpthd_attn_fwd_tc(const void* q, const int32_t* q_idx, int q_rows, const void* k,
                      const void* v, void* o, void* o_resid, float* lse, const void* meta,
                      size_t meta_bytes,
                      int T, int H, int D, int s_local, int cp, int rank, int strategy,
                      float scale_log2, int f16, cudaStream_t s, uint64_t limit_ns,
                      int skip_first_k) {
  using namespace cpthd;
  TcArgs a{};
  a.o = (bf16*)o;
  a.o_resid = (bf16*)o_resid;
  a.lse = lse;
  a.q_idx = q_idx;
  a.q_rows = q_rows;
  a.meta = meta;
  a.meta_bytes = meta_bytes;
  a.T = T; a.H = H; a.s_local = s_local; a.cp = cp; a.rank = rank; a.strategy = strategy;
  a.scale_log2 = scale_log2;
  a.limit_ns = limit_ns ? limit_ns : kWaitLimitNs;
  a.skip_first_k = skip_first_k;
  a.n_steps = 1;
  a.kv_rows = T;
  if (f16) return D == 64 ? launch_fwd_tc<64, true>(q, k, v, a, s) : launch_fwd_tc<128, true>(q, k, v, a, s);
  return D == 64 ? launch_fwd_tc<64, false>(q, k, v, a, s) : launch_fwd_tc<128, false>(q, k, v, a, s);
}

// Internal entry of the ring forward in one pass (arguments validated): rank
// `rank`'s n_steps ring steps, step i attending q_local to the shard of rank
// (rank - i) mod cp (rows s_local * that rank of k_shards / v_shards, the
// ranks' shards side by side), with one online softmax over all of them;
// step_meta holds the steps' cp_size = 1 metadata step_bytes apart; scratch
// holds n_qt ints then (16-aligned) n_qt int2 of the work order.
int cpthd_attn_fwd_ring_tc(const void* q, const void* k_shards, const void* v_shards, void* o,
                           void* o_resid, float* lse, const void* step_meta, size_t step_bytes,
                           int n_steps, int H, int D, int s_local, int cp, int rank, int strategy,
                           float scale_log2, int f16, void* scratch, cudaStream_t s) {
  using namespace cpthd;
  TcArgs a{};
  a.o = (bf16*)o;
  a.o_resid = (bf16*)o_resid;
  a.lse = lse;
  a.meta = step_meta;
  a.meta_bytes = step_bytes;
  a.T = s_local; a.H = H; a.s_local = s_local; a.cp = 1; a.rank = 0; a.strategy = strategy;
  a.scale_log2 = scale_log2;
  a.limit_ns = kWaitLimitNs;
  a.n_steps = n_steps;
  a.step_stride = (int64_t)step_bytes;
  a.ring_rank = rank;
  a.ring_cp = cp;
  a.shard_rows = s_local;
  a.kv_rows = s_local * cp;
  const int n_qt = (int)n_tiles_of(s_local);
  int* tot = reinterpret_cast<int*>(scratch);
  int2* order = reinterpret_cast<int2*>(reinterpret_cast<char*>(scratch) + ring_order_offset(s_local));
  a.rorder = order;
  ring_order_kernel<<<1, kOrdThreads, 0, s>>>(a, tot, order);
  int st = cpthd_host::launch_status();
  if (st != CP_OK || n_qt == 0) return st;
  if (f16) return D == 64 ? launch_fwd_tc<64, true>(q, k_shards, v_shards, a, s)
                          : launch_fwd_tc<128, true>(q, k_shards, v_shards, a, s);
  return D == 64 ? launch_fwd_tc<64, false>(q, k_shards, v_shards, a, s)
                 : launch_fwd_tc<128, false>(q, k_shards, v_shards, a, s);
}

extern "C" int cpthd_status_fwd_tc(int reset) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, cpthd::g_status_fwd_tc, sizeof(int)) != cudaSuccess)
    return CP_ERR_CUDA;
  if (reset) {
    int z = 0;
    if (cudaMemcpyToSymbol(cpthd::g_status_fwd_tc, &z, sizeof(int)) != cudaSuccess)
      return CP_ERR_CUDA;
  }
  return v;
}
