// attn_mma.cu -- causal varlen attention over THD-packed documents, one CP
// rank's local queries against the full (restored) K/V, fwd and bwd.
//
// "[PyTorch] Add no-load-balance THD all-gather CP", §Why / §Scope and
// constraints: causal, no sliding window, document boundaries from the THD
// metadata; DUAL_CHUNK_SWAP's two attention steps per rank are fused into one
// launch here because every local row carries its own global position and
// document start (row tables built by the partition kernel).
//
// The forward runs on the tcgen05 tensor cores (attn_fwd_tc.cu); this file
// holds the entry points and the backward kernels (bf16 in, fp32 accumulate,
// warp-level mma.sync m16n8k16):
//   attn_delta     Delta = rowsum(dO * O) (fp32, [H, s_local])
//   attn_dq_mma    dQ per 64-query tile, iterating its key blocks
//   attn_dkdv_mma  dK/dV per 64-key block, iterating the query tiles that
//                  attend it; each key block has exactly one owner CTA, so the
//                  fp32 read-modify-write accumulation is deterministic
// Key blocks a tile needs come from the segment table: for each segment in
// the tile, keys [doc start, last real query], merged in increasing order.
#include <math.h>

#include <mutex>

#include "common.cuh"

namespace cpthd {

static __device__ int g_status_attn;

namespace {

using bf16 = __nv_bfloat16;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kThreads = 128;  // 4 warps
constexpr int BM = 64;         // query rows per tile (16 per warp)
constexpr int BN = 64;         // keys per block
constexpr int kMaxIv = 2 * BM + 4;

struct AttnArgs {
  const bf16* q;     // [s_local, H, D]
  const bf16* k;     // [T, H, D]
  const bf16* v;     // [T, H, D]
  bf16* o;           // [s_local, H, D]
  float* lse;        // [H, s_local]
  const bf16* dout;  // [s_local, H, D]
  const bf16* out;   // [s_local, H, D]  (forward output, for Delta)
  float* delta;      // [H, s_local]
  bf16* dq;          // [s_local, H, D]
  float* dk;         // [T, H, D] fp32 accumulators
  float* dv;
  const void* meta;
  size_t meta_bytes;
  int T, H, s_local, cp, rank, strategy;
  float scale, scale_log2;
};

// Every kernel first checks that the metadata belongs to this call.
__device__ __forceinline__ bool meta_ok(const AttnArgs& a, const MetaView& m) {
  const MetaHeader* h = m.hdr;
  // the tables must lie inside the caller's buffer
  const bool fits = h->n_segs >= 0 && h->n_segs <= h->max_segs && h->seg_offset == 64 &&
                    (int64_t)h->rows_offset >= 64 + 32 * (int64_t)h->max_segs &&
                    (int64_t)h->rows_offset + 8 * (int64_t)a.s_local <= (int64_t)a.meta_bytes;
  const bool ok = fits && h->magic == kMetaMagic && h->status == 0 && h->s_local == a.s_local &&
                  h->rank == a.rank && h->cp_size == a.cp && h->strategy == a.strategy &&
                  h->total_tokens == a.T;
  if (!ok && threadIdx.x == 0)
    atomicCAS(&g_status_attn, 0, h->status != 0 ? h->status : (int)CP_ERR_METADATA);
  return ok;
}

// cp.async a [64 rows][D] bf16 tile (rows row0.., head h) into a swizzled
// smem tile; rows >= n_rows are zero-filled.
template <int D>
__device__ __forceinline__ void load_tile(uint32_t s_base, const bf16* g, int row0, int n_rows,
                                          int H, int h) {
  constexpr int RC = D / 8;
  for (int c = threadIdx.x; c < 64 * RC; c += kThreads) {
    const int r = c / RC, ch = c % RC;
    const int row = row0 + r;
    const bool ok = row < n_rows;
    const bf16* src = g + ((int64_t)(ok ? row : 0) * H + h) * D + ch * 8;
    cp_async_16(s_base + swz(r, ch, RC), src, ok);
  }
}

// Iterator over the flattened block sequence of a list of intervals.
struct BlockIter {
  const int2* iv;
  int n_iv, i, b;
  __device__ void init(const int2* p, int n) {
    iv = p; n_iv = n; i = 0; b = n > 0 ? p[0].x : 0;
  }
  __device__ void next() {
    if (b < iv[i].y) { ++b; } else { ++i; if (i < n_iv) b = iv[i].x; }
  }
};

__device__ __forceinline__ int total_blocks(const int2* iv, int n) {
  int t = 0;
  for (int i = 0; i < n; ++i) t += iv[i].y - iv[i].x + 1;
  return t;
}

// ---------------------------------------------------------------------------
// backward: Delta = rowsum(dO * O)
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) attn_delta(const AttnArgs a) {
  constexpr int G = D / 8;  // threads per (row, head)
  const int64_t gid = int64_t(blockIdx.x) * 256 + threadIdx.x;
  const int64_t pair = gid / G;  // row * H + head
  const int part = (int)(gid % G);
  const int64_t n_pairs = (int64_t)a.s_local * a.H;
  float acc = 0.f;
  if (pair < n_pairs) {
    const uint4 x = *reinterpret_cast<const uint4*>(a.dout + pair * D + part * 8);
    const uint4 y = *reinterpret_cast<const uint4*>(a.out + pair * D + part * 8);
    const __nv_bfloat162* xp = reinterpret_cast<const __nv_bfloat162*>(&x);
    const __nv_bfloat162* yp = reinterpret_cast<const __nv_bfloat162*>(&y);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 fx = __bfloat1622float2(xp[i]), fy = __bfloat1622float2(yp[i]);
      acc += fx.x * fy.x + fx.y * fy.y;
    }
  }
#pragma unroll
  for (int off = G / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (pair < n_pairs && part == 0) {
    const int64_t row = pair / a.H;
    const int h = (int)(pair % a.H);
    a.delta[(int64_t)h * a.s_local + row] = acc;
  }
}

// ---------------------------------------------------------------------------
// backward: dQ per query tile
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kThreads)
attn_dq_mma(const AttnArgs a) {
  constexpr int RC = D / 8;
  constexpr int TILE = 64 * D * 2;
  extern __shared__ __align__(128) char smem[];
  __shared__ int2 s_iv[kMaxIv];
  __shared__ int s_niv;

  const MetaView m = meta_view(a.meta);
  if (!meta_ok(a, m)) return;
  const int tile = gridDim.x - 1 - blockIdx.x;
  const int h = blockIdx.y;
  const int t0 = tile * BM;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sQ = smem_u32(smem), sO = sQ + TILE;
  const uint32_t sK0 = sQ + 2 * TILE, sV0 = sQ + 4 * TILE;

  if (tid == 0) s_niv = build_kv_intervals(m, t0, min(BM, a.s_local - t0), BN, s_iv, kMaxIv);
  load_tile<D>(sQ, a.q, t0, a.s_local, a.H, h);
  load_tile<D>(sO, a.dout, t0, a.s_local, a.H, h);
  cp_async_commit();
  __syncthreads();

  const int ra = warp * 16 + (lane >> 2), rb = ra + 8;
  const int ta = t0 + ra, tb = t0 + rb;
  const int lo_a = ta < a.s_local ? m.row_lo[ta] : 0, hi_a = ta < a.s_local ? m.row_hi[ta] : -1;
  const int lo_b = tb < a.s_local ? m.row_lo[tb] : 0, hi_b = tb < a.s_local ? m.row_hi[tb] : -1;
  const float lse_a = hi_a >= 0 ? a.lse[(int64_t)h * a.s_local + ta] * kLog2e : 0.f;
  const float lse_b = hi_b >= 0 ? a.lse[(int64_t)h * a.s_local + tb] * kLog2e : 0.f;
  const float dl_a = hi_a >= 0 ? a.delta[(int64_t)h * a.s_local + ta] : 0.f;
  const float dl_b = hi_b >= 0 ? a.delta[(int64_t)h * a.s_local + tb] : 0.f;

  BlockIter it;
  it.init(s_iv, s_niv);
  const int nb = total_blocks(s_iv, s_niv);

  float dq[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) dq[i][0] = dq[i][1] = dq[i][2] = dq[i][3] = 0.f;

  int cur_blk = 0;
  if (nb > 0) {
    cur_blk = it.b;
    load_tile<D>(sK0, a.k, cur_blk * BN, a.T, a.H, h);
    load_tile<D>(sV0, a.v, cur_blk * BN, a.T, a.H, h);
    cp_async_commit();
    it.next();
  }
  const int mi = lane >> 3, l8 = lane & 7;
  for (int n = 0; n < nb; ++n) {
    const int stage = n & 1;
    if (n + 1 < nb) {
      const uint32_t off = (stage ^ 1) * TILE;
      load_tile<D>(sK0 + off, a.k, it.b * BN, a.T, a.H, h);
      load_tile<D>(sV0 + off, a.v, it.b * BN, a.T, a.H, h);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint32_t sK = sK0 + stage * TILE, sV = sV0 + stage * TILE;
    const int j0 = cur_blk * BN;

    float s[BN / 8][4], dp[BN / 8][4];
#pragma unroll
    for (int i = 0; i < BN / 8; ++i) {
      s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
      dp[i][0] = dp[i][1] = dp[i][2] = dp[i][3] = 0.f;
    }
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t qa[4], oa[4];
      ldsm_x4(sQ + swz(warp * 16 + (mi & 1) * 8 + l8, kk * 2 + (mi >> 1), RC), qa[0], qa[1], qa[2], qa[3]);
      ldsm_x4(sO + swz(warp * 16 + (mi & 1) * 8 + l8, kk * 2 + (mi >> 1), RC), oa[0], oa[1], oa[2], oa[3]);
#pragma unroll
      for (int np = 0; np < BN / 16; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(sK + swz(np * 16 + (mi >> 1) * 8 + l8, kk * 2 + (mi & 1), RC), b0, b1, b2, b3);
        mma_16816(s[2 * np], qa, b0, b1);
        mma_16816(s[2 * np + 1], qa, b2, b3);
        ldsm_x4(sV + swz(np * 16 + (mi >> 1) * 8 + l8, kk * 2 + (mi & 1), RC), b0, b1, b2, b3);
        mma_16816(dp[2 * np], oa, b0, b1);
        mma_16816(dp[2 * np + 1], oa, b2, b3);
      }
    }
    // P and dS = P * (dP - Delta)
#pragma unroll
    for (int nt = 0; nt < BN / 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = j0 + nt * 8 + (lane & 3) * 2 + (e & 1);
        const bool ok = e < 2 ? (key >= lo_a && key <= hi_a) : (key >= lo_b && key <= hi_b);
        const float p = ok ? exp2f(s[nt][e] * a.scale_log2 - (e < 2 ? lse_a : lse_b)) : 0.f;
        s[nt][e] = p * (dp[nt][e] - (e < 2 ? dl_a : dl_b));
      }
    }
    // dQ += dS K
#pragma unroll
    for (int kk = 0; kk < BN / 16; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int dd = 0; dd < D / 16; ++dd) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(sK + swz(kk * 16 + (mi & 1) * 8 + l8, dd * 2 + (mi >> 1), RC), b0, b1, b2, b3);
        mma_16816(dq[2 * dd], pa, b0, b1);
        mma_16816(dq[2 * dd + 1], pa, b2, b3);
      }
    }
    __syncthreads();
    cur_blk = it.b;
    it.next();
  }

  const int col = (lane & 3) * 2;
  if (ta < a.s_local) {
    bf16* dst = a.dq + ((int64_t)ta * a.H + h) * D;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt)
      *reinterpret_cast<uint32_t*>(dst + nt * 8 + col) =
          pack_bf16(dq[nt][0] * a.scale, dq[nt][1] * a.scale);
  }
  if (tb < a.s_local) {
    bf16* dst = a.dq + ((int64_t)tb * a.H + h) * D;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt)
      *reinterpret_cast<uint32_t*>(dst + nt * 8 + col) =
          pack_bf16(dq[nt][2] * a.scale, dq[nt][3] * a.scale);
  }
}

// ---------------------------------------------------------------------------
// backward: dK, dV per key block
// ---------------------------------------------------------------------------
constexpr int BQ = 64;  // queries per step of the dK/dV loop

template <int D>
__global__ void __launch_bounds__(kThreads)
attn_dkdv_mma(const AttnArgs a) {
  constexpr int RC = D / 8;
  constexpr int TILE = 64 * D * 2;
  extern __shared__ __align__(128) char smem[];
  __shared__ int2 s_iv[kMaxIv];
  __shared__ int s_niv;
  __shared__ int s_lo[2][BQ], s_hi[2][BQ];
  __shared__ float s_lse[2][BQ], s_dl[2][BQ];

  const MetaView m = meta_view(a.meta);
  if (!meta_ok(a, m)) return;
  const int kb = blockIdx.x;
  const int h = blockIdx.y;
  const int j0 = kb * BN;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sK = smem_u32(smem), sV = sK + TILE;
  const uint32_t sQ0 = sK + 2 * TILE, sO0 = sK + 4 * TILE;

  if (tid == 0) s_niv = build_q_intervals(m, j0, min(j0 + BN, a.T) - 1, BQ, s_iv, kMaxIv);
  __syncthreads();
  const int nb = total_blocks(s_iv, s_niv);
  if (nb == 0) return;  // no query of this rank attends these keys
  BlockIter it;
  it.init(s_iv, s_niv);

  load_tile<D>(sK, a.k, j0, a.T, a.H, h);
  load_tile<D>(sV, a.v, j0, a.T, a.H, h);
  cp_async_commit();

  auto load_qstep = [&](int stage, int qt) {
    const int q0 = qt * BQ;
    load_tile<D>(sQ0 + stage * TILE, a.q, q0, a.s_local, a.H, h);
    load_tile<D>(sO0 + stage * TILE, a.dout, q0, a.s_local, a.H, h);
    if (tid < BQ) {
      const int t = q0 + tid;
      const bool in = t < a.s_local;
      const int hi = in ? m.row_hi[t] : -1;
      s_lo[stage][tid] = in ? m.row_lo[t] : 0;
      s_hi[stage][tid] = hi;
      s_lse[stage][tid] = hi >= 0 ? a.lse[(int64_t)h * a.s_local + t] * kLog2e : 0.f;
      s_dl[stage][tid] = hi >= 0 ? a.delta[(int64_t)h * a.s_local + t] : 0.f;
    }
  };

  float dk[D / 8][4], dv[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) {
    dk[i][0] = dk[i][1] = dk[i][2] = dk[i][3] = 0.f;
    dv[i][0] = dv[i][1] = dv[i][2] = dv[i][3] = 0.f;
  }

  int cur = it.b;
  load_qstep(0, cur);
  cp_async_commit();
  it.next();

  const int mi = lane >> 3, l8 = lane & 7;
  const int key_a = j0 + warp * 16 + (lane >> 2), key_b = key_a + 8;
  for (int n = 0; n < nb; ++n) {
    const int stage = n & 1;
    if (n + 1 < nb) {
      load_qstep(stage ^ 1, it.b);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint32_t sQ = sQ0 + stage * TILE, sO = sO0 + stage * TILE;

    // S^T = K Q^T and dP^T = V dO^T : rows = this warp's 16 keys, cols = queries
    float s[BQ / 8][4], dp[BQ / 8][4];
#pragma unroll
    for (int i = 0; i < BQ / 8; ++i) {
      s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
      dp[i][0] = dp[i][1] = dp[i][2] = dp[i][3] = 0.f;
    }
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t ka[4], va[4];
      ldsm_x4(sK + swz(warp * 16 + (mi & 1) * 8 + l8, kk * 2 + (mi >> 1), RC), ka[0], ka[1], ka[2], ka[3]);
      ldsm_x4(sV + swz(warp * 16 + (mi & 1) * 8 + l8, kk * 2 + (mi >> 1), RC), va[0], va[1], va[2], va[3]);
#pragma unroll
      for (int np = 0; np < BQ / 16; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(sQ + swz(np * 16 + (mi >> 1) * 8 + l8, kk * 2 + (mi & 1), RC), b0, b1, b2, b3);
        mma_16816(s[2 * np], ka, b0, b1);
        mma_16816(s[2 * np + 1], ka, b2, b3);
        ldsm_x4(sO + swz(np * 16 + (mi >> 1) * 8 + l8, kk * 2 + (mi & 1), RC), b0, b1, b2, b3);
        mma_16816(dp[2 * np], va, b0, b1);
        mma_16816(dp[2 * np + 1], va, b2, b3);
      }
    }
    // P^T and dS^T
#pragma unroll
    for (int nt = 0; nt < BQ / 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int qc = nt * 8 + (lane & 3) * 2 + (e & 1);
        const int key = e < 2 ? key_a : key_b;
        const bool ok = key >= s_lo[stage][qc] && key <= s_hi[stage][qc];
        const float p = ok ? exp2f(s[nt][e] * a.scale_log2 - s_lse[stage][qc]) : 0.f;
        s[nt][e] = p;
        dp[nt][e] = p * (dp[nt][e] - s_dl[stage][qc]);
      }
    }
    // dV += P^T dO ; dK += dS^T Q
#pragma unroll
    for (int kk = 0; kk < BQ / 16; ++kk) {
      uint32_t pa[4], da[4];
      pa[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
      da[0] = pack_bf16(dp[2 * kk][0], dp[2 * kk][1]);
      da[1] = pack_bf16(dp[2 * kk][2], dp[2 * kk][3]);
      da[2] = pack_bf16(dp[2 * kk + 1][0], dp[2 * kk + 1][1]);
      da[3] = pack_bf16(dp[2 * kk + 1][2], dp[2 * kk + 1][3]);
#pragma unroll
      for (int dd = 0; dd < D / 16; ++dd) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(sO + swz(kk * 16 + (mi & 1) * 8 + l8, dd * 2 + (mi >> 1), RC), b0, b1, b2, b3);
        mma_16816(dv[2 * dd], pa, b0, b1);
        mma_16816(dv[2 * dd + 1], pa, b2, b3);
        ldsm_x4_t(sQ + swz(kk * 16 + (mi & 1) * 8 + l8, dd * 2 + (mi >> 1), RC), b0, b1, b2, b3);
        mma_16816(dk[2 * dd], da, b0, b1);
        mma_16816(dk[2 * dd + 1], da, b2, b3);
      }
    }
    __syncthreads();
    cur = it.b;
    it.next();
  }
  (void)cur;

  // accumulate this rank's partial into the fp32 accumulators (unique owner)
  const int col = (lane & 3) * 2;
  if (key_a < a.T) {
    float* pk = a.dk + ((int64_t)key_a * a.H + h) * D + col;
    float* pv = a.dv + ((int64_t)key_a * a.H + h) * D + col;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      float2 x = *reinterpret_cast<float2*>(pk + nt * 8);
      x.x += dk[nt][0] * a.scale; x.y += dk[nt][1] * a.scale;
      *reinterpret_cast<float2*>(pk + nt * 8) = x;
      float2 y = *reinterpret_cast<float2*>(pv + nt * 8);
      y.x += dv[nt][0]; y.y += dv[nt][1];
      *reinterpret_cast<float2*>(pv + nt * 8) = y;
    }
  }
  if (key_b < a.T) {
    float* pk = a.dk + ((int64_t)key_b * a.H + h) * D + col;
    float* pv = a.dv + ((int64_t)key_b * a.H + h) * D + col;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      float2 x = *reinterpret_cast<float2*>(pk + nt * 8);
      x.x += dk[nt][2] * a.scale; x.y += dk[nt][3] * a.scale;
      *reinterpret_cast<float2*>(pk + nt * 8) = x;
      float2 y = *reinterpret_cast<float2*>(pv + nt * 8);
      y.x += dv[nt][2]; y.y += dv[nt][3];
      *reinterpret_cast<float2*>(pv + nt * 8) = y;
    }
  }
}

template <typename K>
int launch(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, const AttnArgs& a) {
  // dynamic + static shared memory above 48 KB needs the opt-in attribute
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return CP_ERR_CUDA;
  kernel<<<grid, block, smem, st>>>(a);
  return cpthd_host::launch_status();
}

int common_checks(const void* q, const void* k, const void* v, const void* meta, size_t meta_bytes,
                  int64_t T, int H, int D, int cp, int rank, cp_strategy_t strategy,
                  int64_t* s_local) {
  if (!q || !k || !v || !meta) return CP_ERR_INVALID_ARG;
  if (H < 1 || T < 0 || T > INT32_MAX || cp < 1 || rank < 0 || rank >= cp) return CP_ERR_INVALID_ARG;
  if (strategy != CP_DUAL_CHUNK_SWAP && strategy != CP_NO_LOAD_BALANCE) return CP_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return CP_ERR_UNSUPPORTED;
  if (H > 65535) return CP_ERR_UNSUPPORTED;
  if (T % cp) return CP_ERR_DIVISIBILITY;
  *s_local = T / cp;
  if ((int64_t)T * H * D > ((int64_t)1 << 40)) return CP_ERR_UNSUPPORTED;
  if (meta_bytes < 64) return CP_ERR_WORKSPACE;
  if (!cpthd_host::aligned16(q) || !cpthd_host::aligned16(k) || !cpthd_host::aligned16(v) ||
      !cpthd_host::aligned16(meta))
    return CP_ERR_ALIGNMENT;
  return CP_OK;
}

}  // namespace
}  // namespace cpthd

using namespace cpthd;

extern "C" int cp_attn_fwd(const void* q_local, const void* k_full, const void* v_full,
                           void* o_local, float* lse_local, const void* d_meta, size_t meta_bytes,
                           int64_t total_tokens, int H, int D, int cp_size, int rank,
                           cp_strategy_t strategy, float softmax_scale, void* stream) {
  int64_t s_local = 0;
  int st = common_checks(q_local, k_full, v_full, d_meta, meta_bytes, total_tokens, H, D, cp_size,
                         rank, strategy, &s_local);
  if (st != CP_OK) return st;
  if (!o_local || !lse_local) return CP_ERR_INVALID_ARG;
  if (!cpthd_host::aligned16(o_local) || !cpthd_host::aligned16(lse_local)) return CP_ERR_ALIGNMENT;
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return CP_ERR_INVALID_ARG;
  if (s_local == 0) return CP_OK;
  return cpthd_attn_fwd_tc(q_local, k_full, v_full, o_local, lse_local, d_meta, meta_bytes,
                           (int)total_tokens, H, D, (int)s_local, cp_size, rank, (int)strategy,
                           softmax_scale * kLog2e, cpthd_host::as_stream(stream));
}

extern "C" size_t cp_attn_bwd_workspace_bytes(int64_t s_local, int H) {
  if (s_local < 0 || H < 1) return 0;
  return (size_t)s_local * H * sizeof(float);
}

extern "C" int cp_attn_bwd(const void* q_local, const void* k_full, const void* v_full,
                           const void* o_local, const float* lse_local, const void* do_local,
                           void* dq_local, float* dk_accum, float* dv_accum, const void* d_meta,
                           size_t meta_bytes, int64_t total_tokens, int H, int D, int cp_size,
                           int rank, cp_strategy_t strategy, float softmax_scale,
                           void* d_workspace, size_t workspace_bytes, void* stream) {
  int64_t s_local = 0;
  int st = common_checks(q_local, k_full, v_full, d_meta, meta_bytes, total_tokens, H, D, cp_size,
                         rank, strategy, &s_local);
  if (st != CP_OK) return st;
  if (!o_local || !lse_local || !do_local || !dq_local || !dk_accum || !dv_accum)
    return CP_ERR_INVALID_ARG;
  if (!cpthd_host::aligned16(o_local) || !cpthd_host::aligned16(lse_local) ||
      !cpthd_host::aligned16(do_local) || !cpthd_host::aligned16(dq_local) ||
      !cpthd_host::aligned16(dk_accum) || !cpthd_host::aligned16(dv_accum))
    return CP_ERR_ALIGNMENT;
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return CP_ERR_INVALID_ARG;
  if (s_local == 0) return CP_OK;
  if (!d_workspace || workspace_bytes < cp_attn_bwd_workspace_bytes(s_local, H))
    return CP_ERR_WORKSPACE;
  if (!cpthd_host::aligned16(d_workspace)) return CP_ERR_ALIGNMENT;
  AttnArgs a{};
  a.q = (const bf16*)q_local; a.k = (const bf16*)k_full; a.v = (const bf16*)v_full;
  a.out = (const bf16*)o_local; a.lse = const_cast<float*>(lse_local);
  a.dout = (const bf16*)do_local; a.dq = (bf16*)dq_local; a.dk = dk_accum; a.dv = dv_accum;
  a.delta = (float*)d_workspace; a.meta = d_meta; a.meta_bytes = meta_bytes;
  a.T = (int)total_tokens; a.H = H; a.s_local = (int)s_local; a.cp = cp_size; a.rank = rank;
  a.strategy = (int)strategy; a.scale = softmax_scale; a.scale_log2 = softmax_scale * kLog2e;
  cudaStream_t s = cpthd_host::as_stream(stream);
  const int64_t threads = s_local * H * (D / 8);
  dim3 dgrid((unsigned)((threads + 255) / 256));
  if (D == 64) attn_delta<64><<<dgrid, 256, 0, s>>>(a);
  else attn_delta<128><<<dgrid, 256, 0, s>>>(a);
  if ((st = cpthd_host::launch_status()) != CP_OK) return st;
  dim3 qgrid((unsigned)((s_local + BM - 1) / BM), (unsigned)H);
  const size_t qsmem = (size_t)6 * 64 * D * 2;
  st = D == 64 ? launch(attn_dq_mma<64>, qgrid, kThreads, qsmem, s, a)
               : launch(attn_dq_mma<128>, qgrid, kThreads, qsmem, s, a);
  if (st != CP_OK) return st;
  dim3 kgrid((unsigned)((total_tokens + BN - 1) / BN), (unsigned)H);
  const size_t ksmem = (size_t)6 * 64 * D * 2;
  return D == 64 ? launch(attn_dkdv_mma<64>, kgrid, kThreads, ksmem, s, a)
                 : launch(attn_dkdv_mma<128>, kgrid, kThreads, ksmem, s, a);
}

extern "C" int cpthd_status_attn(int reset) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status_attn, sizeof(int)) != cudaSuccess) return CP_ERR_CUDA;
  if (reset) {
    int z = 0;
    if (cudaMemcpyToSymbol(g_status_attn, &z, sizeof(int)) != cudaSuccess) return CP_ERR_CUDA;
  }
  return v;
}

// ---------------------------------------------------------------------------
// Allocation-free backward: the Delta scratch lives in a fixed device array
// of this translation unit instead of a caller-provided workspace.
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) float g_noalloc_scratch[CP_NOALLOC_MAX_SCRATCH_FLOATS];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device, with that device current, and cached.
int noalloc_scratch(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CP_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return CP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return CP_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return CP_OK;
}

}  // namespace

extern "C" int cp_attn_bwd_noalloc(const void* q_local, const void* k_full, const void* v_full,
                                   const void* o_local, const float* lse_local,
                                   const void* do_local, void* dq_local, float* dk_accum,
                                   float* dv_accum, const void* d_meta, size_t meta_bytes,
                                   int64_t total_tokens, int H, int D, int cp_size, int rank,
                                   cp_strategy_t strategy, float softmax_scale, void* stream) {
  int64_t s_local = 0;
  int st = common_checks(q_local, k_full, v_full, d_meta, meta_bytes, total_tokens, H, D, cp_size,
                         rank, strategy, &s_local);
  if (st != CP_OK) return st;
  if (!o_local || !lse_local || !do_local || !dq_local || !dk_accum || !dv_accum)
    return CP_ERR_INVALID_ARG;
  if (!cpthd_host::aligned16(o_local) || !cpthd_host::aligned16(lse_local) ||
      !cpthd_host::aligned16(do_local) || !cpthd_host::aligned16(dq_local) ||
      !cpthd_host::aligned16(dk_accum) || !cpthd_host::aligned16(dv_accum))
    return CP_ERR_ALIGNMENT;
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return CP_ERR_INVALID_ARG;
  if (s_local * (int64_t)H > (int64_t)CP_NOALLOC_MAX_SCRATCH_FLOATS) return CP_ERR_WORKSPACE;
  if (s_local == 0) return CP_OK;
  float* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != CP_OK) return st;
  AttnArgs a{};
  a.q = (const bf16*)q_local; a.k = (const bf16*)k_full; a.v = (const bf16*)v_full;
  a.out = (const bf16*)o_local; a.lse = const_cast<float*>(lse_local);
  a.dout = (const bf16*)do_local; a.dq = (bf16*)dq_local; a.dk = dk_accum; a.dv = dv_accum;
  a.delta = scratch; a.meta = d_meta; a.meta_bytes = meta_bytes;
  a.T = (int)total_tokens; a.H = H; a.s_local = (int)s_local; a.cp = cp_size; a.rank = rank;
  a.strategy = (int)strategy; a.scale = softmax_scale; a.scale_log2 = softmax_scale * kLog2e;
  cudaStream_t s = cpthd_host::as_stream(stream);
  const int64_t threads = s_local * H * (D / 8);
  dim3 dgrid((unsigned)((threads + 255) / 256));
  if (D == 64) attn_delta<64><<<dgrid, 256, 0, s>>>(a);
  else attn_delta<128><<<dgrid, 256, 0, s>>>(a);
  if ((st = cpthd_host::launch_status()) != CP_OK) return st;
  dim3 qgrid((unsigned)((s_local + BM - 1) / BM), (unsigned)H);
  const size_t qsmem = (size_t)6 * 64 * D * 2;
  st = D == 64 ? launch(attn_dq_mma<64>, qgrid, kThreads, qsmem, s, a)
               : launch(attn_dq_mma<128>, qgrid, kThreads, qsmem, s, a);
  if (st != CP_OK) return st;
  dim3 kgrid((unsigned)((total_tokens + BN - 1) / BN), (unsigned)H);
  const size_t ksmem = (size_t)6 * 64 * D * 2;
  return D == 64 ? launch(attn_dkdv_mma<64>, kgrid, kThreads, ksmem, s, a)
                 : launch(attn_dkdv_mma<128>, kgrid, kThreads, ksmem, s, a);
}
