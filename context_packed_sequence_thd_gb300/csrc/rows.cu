// rows.cu -- bandwidth-bound THD row kernels: gather / scatter (the
// index_select restore and unrestore of "[PyTorch] Add no-load-balance THD
// all-gather CP", §Sequence Diagram), the fp32 -> bf16 emulated reduce-scatter
// epilogue of dK/dV, and the gated gradient tail-zeroing of "THD P2P
// context-parallel regression when padded cu_seqlens are value-equal but not
// object-identical" (§Describe the bug, §Expected behavior).
//
// Also the all-to-all exchange of the a2a comm type (see a2a_kernel), and the
// gather that converts bf16 rows to fp16 tensor-core operands.
//
// Design: one warp moves one row at a time; lanes stride over the row's
// 16-byte chunks with several independent loads in flight before the stores
// (rows are 256 B .. 10 KB).  Up to four tensors share one index load and one
// launch.  The grid is a multiple of the SM count, each CTA loops over rows.
#include "common.cuh"

namespace cpthd {

static __device__ int g_status_rows;

namespace {

constexpr int kMaxTensors = 4;
constexpr int kRowThreads = 512;
constexpr int kUnroll = 4;

struct Ptrs {
  const uint4* src[kMaxTensors];
  uint4* dst[kMaxTensors];
};

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void copy_row(const uint4* __restrict__ s, uint4* __restrict__ d,
                                         int chunks, int lane) {
  int c = lane;
  for (; c + 32 * (kUnroll - 1) < chunks; c += 32 * kUnroll) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = ld_stream(s + c + 32 * u);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) d[c + 32 * u] = v[u];
  }
  for (; c < chunks; c += 32) d[c] = ld_stream(s + c);
}

// 16 bytes of bf16 -> 16 bytes of fp16 (round to nearest).  A finite value
// beyond the fp16 range becomes +-65504 and is reported; infinities and NaN
// keep their meaning.
__device__ __forceinline__ uint4 bf16x8_to_f16(uint4 v, bool& out_of_range) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float a = __uint_as_float(w[i] << 16), b = __uint_as_float(w[i] & 0xFFFF0000u);
    if (fabsf(a) > 65504.f && fabsf(a) != INFINITY) { out_of_range = true; a = copysignf(65504.f, a); }
    if (fabsf(b) > 65504.f && fabsf(b) != INFINITY) { out_of_range = true; b = copysignf(65504.f, b); }
    __half2 h = __floats2half2_rn(a, b);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ void copy_row_f16(const uint4* __restrict__ s, uint4* __restrict__ d,
                                             int chunks, int lane, bool& oor) {
  int c = lane;
  for (; c + 32 * (kUnroll - 1) < chunks; c += 32 * kUnroll) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = ld_stream(s + c + 32 * u);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) d[c + 32 * u] = bf16x8_to_f16(v[u], oor);
  }
  for (; c < chunks; c += 32) d[c] = bf16x8_to_f16(ld_stream(s + c), oor);
}

// mode 0: dst[i] = src[idx[i]]; mode 1: dst[idx[i]] = src[i];
// mode 2: dst[i] = fp16(src[idx ? idx[i] : i]) (bf16 source rows)
template <int MODE>
__global__ void __launch_bounds__(kRowThreads)
rows_kernel(Ptrs p, int n_tensors, const int32_t* __restrict__ idx, int64_t n_rows,
            int64_t bound_rows, int chunks) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t(blockIdx.x) * kRowThreads + threadIdx.x) >> 5;
  const int64_t n_warps = (int64_t(gridDim.x) * kRowThreads) >> 5;
  bool oor = false;
  for (int64_t i = warp; i < n_rows; i += n_warps) {
    const int64_t j = (MODE == 2 && !idx) ? i : idx[i];
    if (j < 0 || j >= bound_rows) {
      if (lane == 0) atomicCAS(&g_status_rows, 0, CP_ERR_INVALID_ARG);
      continue;
    }
    const int64_t si = MODE == 1 ? i : j;
    const int64_t di = MODE == 1 ? j : i;
    for (int k = 0; k < n_tensors; ++k) {
      if (MODE == 2)
        copy_row_f16(p.src[k] + si * chunks, p.dst[k] + di * chunks, chunks, lane, oor);
      else
        copy_row(p.src[k] + si * chunks, p.dst[k] + di * chunks, chunks, lane);
    }
  }
  if (MODE == 2 && __any_sync(0xffffffffu, oor) && lane == 0)
    atomicCAS(&g_status_rows, 0, CP_ERR_RANGE);
}

// All-to-all exchange of the a2a comm type ("[PyTorch] Extend no-load-balance
// CP to the a2a comm type", ¶1-2 and §Diagram), every rank on one GPU.  The
// sequence side is the rank-concatenated buffer [T, H, D] (rank r's token
// shard is rows [r*s_local, (r+1)*s_local)); the head side is cp buffers
// [T, H/cp, D] side by side (rank r: all tokens in original order, heads
// [r*H/cp, (r+1)*H/cp)).  Token g of the head side lives at sequence-side row
// perm[g] (the restore index under DUAL_CHUNK_SWAP, so the dual-chunk reorder
// is part of the same pass), or row g when perm is null (flat sharding: the
// rank-concatenated order already is the original order).
// DIR 0 (seq -> head): head[r][g] = seq[perm(g)][slice r]
// DIR 1 (head -> seq): seq[perm(g)][slice r] = head[r][g]
// One warp per (token, rank) unit, units token-major so that consecutive
// warps move consecutive slices of one sequence-side row.
template <int DIR>
__global__ void __launch_bounds__(kRowThreads)
a2a_kernel(Ptrs p, int n_tensors, const int32_t* __restrict__ perm, int64_t T, int cp,
           int slice_chunks, int row_chunks) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t(blockIdx.x) * kRowThreads + threadIdx.x) >> 5;
  const int64_t n_warps = (int64_t(gridDim.x) * kRowThreads) >> 5;
  const int64_t units = T * cp;
  for (int64_t u = warp; u < units; u += n_warps) {
    const int64_t g = u / cp;
    const int r = (int)(u - g * cp);
    const int64_t pos = perm ? (int64_t)perm[g] : g;
    if (pos < 0 || pos >= T) {
      if (lane == 0) atomicCAS(&g_status_rows, 0, CP_ERR_INVALID_ARG);
      continue;
    }
    const int64_t seq_off = pos * row_chunks + (int64_t)r * slice_chunks;
    const int64_t head_off = ((int64_t)r * T + g) * slice_chunks;
    for (int k = 0; k < n_tensors; ++k) {
      if (DIR == 0)
        copy_row(p.src[k] + seq_off, p.dst[k] + head_off, slice_chunks, lane);
      else
        copy_row(p.src[k] + head_off, p.dst[k] + seq_off, slice_chunks, lane);
    }
  }
}

struct AccPtrs {
  const float4* src[kMaxTensors];
  uint2* dst[kMaxTensors];
};

// dst[t] = bf16(accum[idx ? idx[t] : row0 + t]); a row is `quads` float4's.
__global__ void __launch_bounds__(kRowThreads)
accum_cast_kernel(AccPtrs p, int n_tensors, const int32_t* __restrict__ idx, int64_t row0,
                  int64_t n_rows, int64_t accum_rows, int quads) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t(blockIdx.x) * kRowThreads + threadIdx.x) >> 5;
  const int64_t n_warps = (int64_t(gridDim.x) * kRowThreads) >> 5;
  for (int64_t t = warp; t < n_rows; t += n_warps) {
    const int64_t j = idx ? (int64_t)idx[t] : row0 + t;
    if (j < 0 || j >= accum_rows) {
      if (lane == 0) atomicCAS(&g_status_rows, 0, CP_ERR_INVALID_ARG);
      continue;
    }
    for (int k = 0; k < n_tensors; ++k) {
      const float4* s = p.src[k] + j * quads;
      uint2* d = p.dst[k] + t * quads;
      int c = lane;
      for (; c + 32 * (kUnroll - 1) < quads; c += 32 * kUnroll) {
        float4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) v[u] = __ldcs(s + c + 32 * u);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
          d[c + 32 * u] = make_uint2(pack_bf16(v[u].x, v[u].y), pack_bf16(v[u].z, v[u].w));
      }
      for (; c < quads; c += 32) {
        float4 v = __ldcs(s + c);
        d[c] = make_uint2(pack_bf16(v.x, v.y), pack_bf16(v.z, v.w));
      }
    }
  }
}

struct ZeroPtrs {
  uint4* dst[kMaxTensors];
};

__global__ void __launch_bounds__(kRowThreads)
zero_tail_kernel(ZeroPtrs p, int n_tensors, int64_t rows, int64_t valid_end,
                 const int32_t* __restrict__ d_valid_end, int chunks) {
  const int64_t ve = d_valid_end ? (int64_t)*d_valid_end : valid_end;
  if (ve >= rows) return;  // no tail: nothing to clear
  const int64_t begin = max((int64_t)0, ve) * chunks;
  const int64_t total = rows * chunks;
  const int64_t stride = int64_t(gridDim.x) * kRowThreads;
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int k = 0; k < n_tensors; ++k)
    for (int64_t c = begin + int64_t(blockIdx.x) * kRowThreads + threadIdx.x; c < total; c += stride)
      p.dst[k][c] = z;
}

int grid_for(int64_t rows_of_work, int warps_per_row_unit) {
  const int sms = cpthd_host::sm_count();
  (void)warps_per_row_unit;
  const int64_t warps = kRowThreads / 32;
  int64_t want = (rows_of_work + warps - 1) / warps;
  int64_t cap = (int64_t)sms * (2048 / kRowThreads);  // one full wave of resident CTAs
  if (want > cap) want = cap;
  if (want < 1) want = 1;
  return (int)want;
}

int validate_rows(const void* const* a, const void* const* b, int n, int64_t n_rows,
                  int64_t row_bytes) {
  if (!a || !b || n < 1 || n > kMaxTensors || n_rows < 0 || row_bytes <= 0)
    return CP_ERR_INVALID_ARG;
  if (row_bytes % 16) return CP_ERR_ALIGNMENT;
  for (int k = 0; k < n; ++k) {
    if (!a[k] || !b[k]) return CP_ERR_INVALID_ARG;
    if (!cpthd_host::aligned16(a[k]) || !cpthd_host::aligned16(b[k])) return CP_ERR_ALIGNMENT;
  }
  if (row_bytes / 16 > INT32_MAX) return CP_ERR_UNSUPPORTED;
  return CP_OK;
}

}  // namespace
}  // namespace cpthd

using namespace cpthd;

static int rows_op(int mode, const void* const* src, void* const* dst, int n, const int32_t* idx,
                   int64_t n_rows, int64_t bound_rows, int64_t row_bytes, void* stream) {
  int st = validate_rows(src, reinterpret_cast<const void* const*>(dst), n, n_rows, row_bytes);
  if (st != CP_OK) return st;
  if ((!idx && mode != 2) || bound_rows < 0) return CP_ERR_INVALID_ARG;
  if (!idx && bound_rows < n_rows) return CP_ERR_INVALID_ARG;
  if (n_rows == 0) return CP_OK;
  Ptrs p{};
  for (int k = 0; k < n; ++k) {
    p.src[k] = reinterpret_cast<const uint4*>(src[k]);
    p.dst[k] = reinterpret_cast<uint4*>(dst[k]);
  }
  const int chunks = (int)(row_bytes / 16);
  const int grid = grid_for(n_rows, 1);
  cudaStream_t s = cpthd_host::as_stream(stream);
  if (mode == 0)
    rows_kernel<0><<<grid, kRowThreads, 0, s>>>(p, n, idx, n_rows, bound_rows, chunks);
  else if (mode == 1)
    rows_kernel<1><<<grid, kRowThreads, 0, s>>>(p, n, idx, n_rows, bound_rows, chunks);
  else
    rows_kernel<2><<<grid, kRowThreads, 0, s>>>(p, n, idx, n_rows, bound_rows, chunks);
  return cpthd_host::launch_status();
}

extern "C" int cp_thd_gather(const void* const* d_src, void* const* d_dst, int n_tensors,
                             const int32_t* d_idx, int64_t n_rows, int64_t src_rows,
                             int64_t row_bytes, void* stream) {
  return rows_op(0, d_src, d_dst, n_tensors, d_idx, n_rows, src_rows, row_bytes, stream);
}

extern "C" int cp_thd_gather_f16(const void* const* d_src, void* const* d_dst, int n_tensors,
                                 const int32_t* d_idx, int64_t n_rows, int64_t src_rows,
                                 int64_t row_bytes, void* stream) {
  return rows_op(2, d_src, d_dst, n_tensors, d_idx, n_rows, src_rows, row_bytes, stream);
}

extern "C" int cp_thd_scatter(const void* const* d_src, void* const* d_dst, int n_tensors,
                              const int32_t* d_idx, int64_t n_rows, int64_t dst_rows,
                              int64_t row_bytes, void* stream) {
  return rows_op(1, d_src, d_dst, n_tensors, d_idx, n_rows, dst_rows, row_bytes, stream);
}

extern "C" int cp_reduce_scatter_emul(const float* const* d_accum, void* const* d_dst,
                                      int n_tensors, const int32_t* d_idx, int64_t row0,
                                      int64_t n_rows, int64_t accum_rows, int H, int D,
                                      void* stream) {
  if (H < 1 || D < 1 || (H * (int64_t)D) % 8) return CP_ERR_ALIGNMENT;
  int st = validate_rows(reinterpret_cast<const void* const*>(d_accum),
                         reinterpret_cast<const void* const*>(d_dst), n_tensors, n_rows,
                         (int64_t)H * D * 2);
  if (st != CP_OK) return st;
  if (accum_rows < 0 || row0 < 0) return CP_ERR_INVALID_ARG;
  if (!d_idx && row0 + n_rows > accum_rows) return CP_ERR_INVALID_ARG;
  if (n_rows == 0) return CP_OK;
  AccPtrs p{};
  for (int k = 0; k < n_tensors; ++k) {
    p.src[k] = reinterpret_cast<const float4*>(d_accum[k]);
    p.dst[k] = reinterpret_cast<uint2*>(d_dst[k]);
  }
  const int quads = (int)((int64_t)H * D / 4);
  accum_cast_kernel<<<grid_for(n_rows, 1), kRowThreads, 0, cpthd_host::as_stream(stream)>>>(
      p, n_tensors, d_idx, row0, n_rows, accum_rows, quads);
  return cpthd_host::launch_status();
}

extern "C" int cp_zero_tail(void* const* d_rows, int n_tensors, int64_t rows, int64_t row_bytes,
                            int64_t valid_end, const int32_t* d_valid_end, void* stream,
                            int* launched) {
  if (launched) *launched = 0;
  int st = validate_rows(reinterpret_cast<const void* const*>(d_rows),
                         reinterpret_cast<const void* const*>(d_rows), n_tensors, rows,
                         row_bytes);
  if (st != CP_OK) return st;
  if (valid_end < 0 && !d_valid_end) return CP_ERR_INVALID_ARG;
  if (valid_end > rows) return CP_ERR_INVALID_ARG;
  if (valid_end >= 0 && valid_end == rows) return CP_OK;  // gated: no tail, no launch
  ZeroPtrs p{};
  for (int k = 0; k < n_tensors; ++k) p.dst[k] = reinterpret_cast<uint4*>(d_rows[k]);
  const int chunks = (int)(row_bytes / 16);
  int64_t tail_rows = valid_end >= 0 ? rows - valid_end : rows;
  int64_t work = tail_rows * chunks;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t grid = (work + kRowThreads - 1) / kRowThreads;
  if (grid > (int64_t)sms * 4) grid = (int64_t)sms * 4;
  if (grid < 1) grid = 1;
  zero_tail_kernel<<<(int)grid, kRowThreads, 0, cpthd_host::as_stream(stream)>>>(
      p, n_tensors, rows, valid_end, valid_end >= 0 ? nullptr : d_valid_end, chunks);
  if (launched) *launched = 1;
  return cpthd_host::launch_status();
}

extern "C" int cp_a2a_exchange(const void* const* d_src, void* const* d_dst, int n_tensors,
                               const int32_t* d_perm, int64_t total_tokens, int cp_size, int H,
                               int D, cp_a2a_dir_t dir, void* stream) {
  if (cp_size < 1 || H < 1 || D < 1 || H % cp_size) return CP_ERR_INVALID_ARG;
  if (dir != CP_A2A_SEQ_TO_HEAD && dir != CP_A2A_HEAD_TO_SEQ) return CP_ERR_INVALID_ARG;
  if (total_tokens < 0 || total_tokens > INT32_MAX) return CP_ERR_INVALID_ARG;
  const int64_t slice_bytes = (int64_t)(H / cp_size) * D * 2;
  int st = validate_rows(d_src, reinterpret_cast<const void* const*>(d_dst), n_tensors,
                         total_tokens, slice_bytes);
  if (st != CP_OK) return st;
  if (total_tokens == 0) return CP_OK;
  Ptrs p{};
  for (int k = 0; k < n_tensors; ++k) {
    p.src[k] = reinterpret_cast<const uint4*>(d_src[k]);
    p.dst[k] = reinterpret_cast<uint4*>(d_dst[k]);
  }
  const int slice_chunks = (int)(slice_bytes / 16);
  const int row_chunks = slice_chunks * cp_size;
  const int grid = grid_for(total_tokens * cp_size, 1);
  cudaStream_t s = cpthd_host::as_stream(stream);
  if (dir == CP_A2A_SEQ_TO_HEAD)
    a2a_kernel<0><<<grid, kRowThreads, 0, s>>>(p, n_tensors, d_perm, total_tokens, cp_size,
                                                slice_chunks, row_chunks);
  else
    a2a_kernel<1><<<grid, kRowThreads, 0, s>>>(p, n_tensors, d_perm, total_tokens, cp_size,
                                                slice_chunks, row_chunks);
  return cpthd_host::launch_status();
}

extern "C" int cpthd_status_rows(int reset) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status_rows, sizeof(int)) != cudaSuccess) return CP_ERR_CUDA;
  if (reset) {
    int z = 0;
    if (cudaMemcpyToSymbol(g_status_rows, &z, sizeof(int)) != cudaSuccess) return CP_ERR_CUDA;
  }
  return v;
}
