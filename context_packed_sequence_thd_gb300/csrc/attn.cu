// attn.cu -- entry points of the causal varlen attention of one CP rank
// (cp_attn_fwd, cp_attn_bwd, cp_attn_bwd_noalloc) and the Delta kernel of the
// backward.
//
// "[PyTorch] Add no-load-balance THD all-gather CP", §Why / §Scope and
// constraints: causal, no sliding window, document boundaries from the THD
// metadata; DUAL_CHUNK_SWAP's two attention steps per rank are fused into one
// launch here because every local row carries its own global position and
// document start (row tables built by the partition kernel).
//
// The forward and the dQ / dK-dV backward kernels run on the tcgen05 tensor
// cores (attn_fwd_tc.cu, attn_bwd_tc.cu).  This file holds argument
// validation and
//   attn_delta  Delta = rowsum(dO * O) (fp32, [H, s_local]), the backward's
//               only scratch.
#include <math.h>

#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace cpthd {

static __device__ int g_status_attn;

namespace {

using bf16 = __nv_bfloat16;
constexpr float kLog2e = 1.4426950408889634f;

struct AttnArgs {
  const bf16* q;     // [s_local, H, D]
  const bf16* k;     // [T, H, D]
  const bf16* v;     // [T, H, D]
  bf16* o;           // [s_local, H, D]
  float* lse;        // [H, s_local]
  const bf16* dout;  // [s_local, H, D]
  const bf16* out;   // [s_local, H, D]  (forward output, for Delta)
  const bf16* out_resid;  // nullable: O - bf16(O) from the forward, rounded to bf16
  float* delta;      // [H, s_local]
  bf16* dq;          // [s_local, H, D]
  float* dk;         // [T, H, D] fp32 accumulators
  float* dv;
  const void* meta;
  size_t meta_bytes;
  int T, H, s_local, cp, rank, strategy;
  float scale, scale_log2;
};

// ---------------------------------------------------------------------------
// backward: Delta = rowsum(dO * O)   (dO of the operand type, O bf16)
// ---------------------------------------------------------------------------
template <int D, bool F16>
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
    const uint4 z = a.out_resid ? *reinterpret_cast<const uint4*>(a.out_resid + pair * D + part * 8)
                                : make_uint4(0, 0, 0, 0);
    const __nv_bfloat162* xp = reinterpret_cast<const __nv_bfloat162*>(&x);
    const __nv_bfloat162* yp = reinterpret_cast<const __nv_bfloat162*>(&y);
    const __nv_bfloat162* zp = reinterpret_cast<const __nv_bfloat162*>(&z);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      // O to about 16 bits: the bf16 output plus its rounding remainder (exact in fp32)
      const float2 fx = F16 ? __half22float2(reinterpret_cast<const __half2*>(&x)[i])
                            : __bfloat1622float2(xp[i]);
      const float2 fy = __bfloat1622float2(yp[i]), fz = __bfloat1622float2(zp[i]);
      acc += fx.x * (fy.x + fz.x) + fx.y * (fy.y + fz.y);
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

int launch_delta(const AttnArgs& a, int D, int f16, cudaStream_t s) {
  const int64_t threads = (int64_t)a.s_local * a.H * (D / 8);
  dim3 dgrid((unsigned)((threads + 255) / 256));
  if (D == 64) {
    if (f16) attn_delta<64, true><<<dgrid, 256, 0, s>>>(a);
    else attn_delta<64, false><<<dgrid, 256, 0, s>>>(a);
  } else {
    if (f16) attn_delta<128, true><<<dgrid, 256, 0, s>>>(a);
    else attn_delta<128, false><<<dgrid, 256, 0, s>>>(a);
  }
  return cpthd_host::launch_status();
}

int check_dtype(cp_dtype_t dtype) {
  return (dtype == CP_OPERAND_BF16 || dtype == CP_OPERAND_F16) ? CP_OK : CP_ERR_INVALID_ARG;
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
                           void* o_local, void* o_resid_local, float* lse_local,
                           const void* d_meta, size_t meta_bytes, int64_t total_tokens, int H,
                           int D, int cp_size, int rank, cp_strategy_t strategy,
                           float softmax_scale, cp_dtype_t operand_dtype, void* stream) {
  int64_t s_local = 0;
  int st = common_checks(q_local, k_full, v_full, d_meta, meta_bytes, total_tokens, H, D, cp_size,
                         rank, strategy, &s_local);
  if (st != CP_OK) return st;
  if ((st = check_dtype(operand_dtype)) != CP_OK) return st;
  if (!o_local || !lse_local) return CP_ERR_INVALID_ARG;
  if (!cpthd_host::aligned16(o_local) || !cpthd_host::aligned16(lse_local) ||
      !cpthd_host::aligned16(o_resid_local))
    return CP_ERR_ALIGNMENT;
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return CP_ERR_INVALID_ARG;
  if (s_local == 0) return CP_OK;
  return cpthd_attn_fwd_tc(q_local, nullptr, 0, k_full, v_full, o_local, o_resid_local, lse_local,
                           d_meta, meta_bytes, (int)total_tokens, H, D, (int)s_local, cp_size,
                           rank, (int)strategy, softmax_scale * kLog2e, (int)operand_dtype,
                           cpthd_host::as_stream(stream));
}

extern "C" int cp_attn_fwd_gather(const void* q_src, int64_t src_rows, const int32_t* d_idx,
                                  const void* k_full, const void* v_full, void* o_local,
                                  void* o_resid_local, float* lse_local, const void* d_meta,
                                  size_t meta_bytes, int64_t total_tokens, int H, int D,
                                  int cp_size, int rank, cp_strategy_t strategy,
                                  float softmax_scale, cp_dtype_t operand_dtype, void* stream) {
  int64_t s_local = 0;
  int st = common_checks(q_src, k_full, v_full, d_meta, meta_bytes, total_tokens, H, D, cp_size,
                         rank, strategy, &s_local);
  if (st != CP_OK) return st;
  if ((st = check_dtype(operand_dtype)) != CP_OK) return st;
  if (!o_local || !lse_local || !d_idx) return CP_ERR_INVALID_ARG;
  if (src_rows < 1 || src_rows > INT32_MAX) return CP_ERR_INVALID_ARG;
  if (!cpthd_host::aligned16(o_local) || !cpthd_host::aligned16(lse_local) ||
      !cpthd_host::aligned16(o_resid_local) || (reinterpret_cast<uintptr_t>(d_idx) & 3u))
    return CP_ERR_ALIGNMENT;
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return CP_ERR_INVALID_ARG;
  if (s_local == 0) return CP_OK;
  return cpthd_attn_fwd_tc(q_src, d_idx, (int)src_rows, k_full, v_full, o_local, o_resid_local,
                           lse_local, d_meta, meta_bytes, (int)total_tokens, H, D, (int)s_local,
                           cp_size, rank, (int)strategy, softmax_scale * kLog2e,
                           (int)operand_dtype, cpthd_host::as_stream(stream));
}

// Failure-detection test hook (not part of the ABI header): cp_attn_fwd
// with every mbarrier wait bounded by limit_ns and the first K tile of CTA 0
// never loaded, so that the wait for it runs out.  The CTA then drains its
// copies, frees its tensor memory and returns; the device status word reads
// CP_ERR_TIMEOUT and the context stays usable.  Nothing else sets the flag.
extern "C" int cpthd_test_attn_fwd_timeout(const void* q_local, const void* k_full,
                                           const void* v_full, void* o_local, float* lse_local,
                                           const void* d_meta, size_t meta_bytes,
                                           int64_t total_tokens, int H, int D, int cp_size,
                                           int rank, cp_strategy_t strategy, float softmax_scale,
                                           cp_dtype_t operand_dtype, uint64_t limit_ns,
                                           void* stream) {
  int64_t s_local = 0;
  int st = common_checks(q_local, k_full, v_full, d_meta, meta_bytes, total_tokens, H, D, cp_size,
                         rank, strategy, &s_local);
  if (st != CP_OK) return st;
  if (!o_local || !lse_local) return CP_ERR_INVALID_ARG;
  if (!cpthd_host::aligned16(o_local) || !cpthd_host::aligned16(lse_local)) return CP_ERR_ALIGNMENT;
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return CP_ERR_INVALID_ARG;
  if (s_local == 0 || limit_ns == 0 || check_dtype(operand_dtype) != CP_OK)
    return CP_ERR_INVALID_ARG;
  return cpthd_attn_fwd_tc(q_local, nullptr, 0, k_full, v_full, o_local, nullptr, lse_local,
                           d_meta, meta_bytes, (int)total_tokens, H, D, (int)s_local, cp_size,
                           rank, (int)strategy, softmax_scale * kLog2e, (int)operand_dtype,
                           cpthd_host::as_stream(stream), limit_ns, 1);
}

extern "C" size_t cp_attn_fwd_ring_workspace_bytes(int64_t s_local) {
  if (s_local < 0) return 0;
  return ring_scratch_bytes(s_local);
}

extern "C" int cp_attn_fwd_ring(const void* q_local, const void* k_shards, const void* v_shards,
                                void* o_local, void* o_resid_local, float* lse_local,
                                const void* d_step_meta, size_t step_bytes, int n_steps,
                                int64_t s_local, int H, int D, int cp_size, int rank,
                                cp_strategy_t strategy, float softmax_scale,
                                cp_dtype_t operand_dtype, void* d_workspace,
                                size_t workspace_bytes, void* stream) {
  if (check_dtype(operand_dtype) != CP_OK) return CP_ERR_INVALID_ARG;
  if (!q_local || !k_shards || !v_shards || !o_local || !lse_local || !d_step_meta)
    return CP_ERR_INVALID_ARG;
  if (H < 1 || cp_size < 1 || rank < 0 || rank >= cp_size || n_steps < 1 || n_steps > cp_size ||
      s_local < 0 || s_local * cp_size > INT32_MAX)
    return CP_ERR_INVALID_ARG;
  if (strategy != CP_DUAL_CHUNK_SWAP && strategy != CP_NO_LOAD_BALANCE) return CP_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return CP_ERR_UNSUPPORTED;
  if (H > 65535 || (int64_t)s_local * cp_size * H * D > ((int64_t)1 << 40)) return CP_ERR_UNSUPPORTED;
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return CP_ERR_INVALID_ARG;
  if (step_bytes < 64) return CP_ERR_WORKSPACE;
  if (step_bytes % 16) return CP_ERR_ALIGNMENT;
  if (!cpthd_host::aligned16(q_local) || !cpthd_host::aligned16(k_shards) ||
      !cpthd_host::aligned16(v_shards) || !cpthd_host::aligned16(o_local) ||
      !cpthd_host::aligned16(o_resid_local) || !cpthd_host::aligned16(lse_local) ||
      !cpthd_host::aligned16(d_step_meta))
    return CP_ERR_ALIGNMENT;
  if (s_local == 0) return CP_OK;
  if (!d_workspace || workspace_bytes < ring_scratch_bytes(s_local)) return CP_ERR_WORKSPACE;
  if (!cpthd_host::aligned16(d_workspace)) return CP_ERR_ALIGNMENT;
  return cpthd_attn_fwd_ring_tc(q_local, k_shards, v_shards, o_local, o_resid_local, lse_local,
                                d_step_meta, step_bytes, n_steps, H, D, (int)s_local, cp_size,
                                rank, (int)strategy, softmax_scale * kLog2e, (int)operand_dtype,
                                d_workspace, cpthd_host::as_stream(stream));
}

extern "C" size_t cp_attn_bwd_workspace_bytes(int64_t s_local, int H) {
  if (s_local < 0 || H < 1) return 0;
  return (size_t)s_local * H * sizeof(float);
}

extern "C" int cp_attn_bwd_ex(const void* q_local, const void* k_full, const void* v_full,
                              const void* o_local, const void* o_resid_local,
                              const float* lse_local, const void* do_local,
                              void* dq_local, float* dk_accum, float* dv_accum, const void* d_meta,
                              size_t meta_bytes, int64_t total_tokens, int H, int D, int cp_size,
                              int rank, cp_strategy_t strategy, float softmax_scale,
                              cp_dtype_t operand_dtype, cp_bwd_mode_t mode, void* d_workspace,
                              size_t workspace_bytes, void* stream) {
  const int m = (int)mode;
  if ((m & ~7) != 0 || (m & 6) == 6) return CP_ERR_INVALID_ARG;
  if (check_dtype(operand_dtype) != CP_OK) return CP_ERR_INVALID_ARG;
  int64_t s_local = 0;
  int st = common_checks(q_local, k_full, v_full, d_meta, meta_bytes, total_tokens, H, D, cp_size,
                         rank, strategy, &s_local);
  if (st != CP_OK) return st;
  if (!o_local || !lse_local || !do_local || !dq_local || !dk_accum || !dv_accum)
    return CP_ERR_INVALID_ARG;
  if (!cpthd_host::aligned16(o_local) || !cpthd_host::aligned16(lse_local) ||
      !cpthd_host::aligned16(do_local) || !cpthd_host::aligned16(dq_local) ||
      !cpthd_host::aligned16(dk_accum) || !cpthd_host::aligned16(dv_accum) ||
      !cpthd_host::aligned16(o_resid_local))
    return CP_ERR_ALIGNMENT;
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return CP_ERR_INVALID_ARG;
  if (s_local == 0) return CP_OK;
  if (!d_workspace || workspace_bytes < cp_attn_bwd_workspace_bytes(s_local, H))
    return CP_ERR_WORKSPACE;
  if (!cpthd_host::aligned16(d_workspace)) return CP_ERR_ALIGNMENT;
  AttnArgs a{};
  a.q = (const bf16*)q_local; a.k = (const bf16*)k_full; a.v = (const bf16*)v_full;
  a.out = (const bf16*)o_local; a.out_resid = (const bf16*)o_resid_local;
  a.lse = const_cast<float*>(lse_local);
  a.dout = (const bf16*)do_local; a.dq = (bf16*)dq_local; a.dk = dk_accum; a.dv = dv_accum;
  a.delta = (float*)d_workspace; a.meta = d_meta; a.meta_bytes = meta_bytes;
  a.T = (int)total_tokens; a.H = H; a.s_local = (int)s_local; a.cp = cp_size; a.rank = rank;
  a.strategy = (int)strategy; a.scale = softmax_scale; a.scale_log2 = softmax_scale * kLog2e;
  cudaStream_t s = cpthd_host::as_stream(stream);
  if ((st = launch_delta(a, D, (int)operand_dtype, s)) != CP_OK) return st;
  return cpthd_attn_bwd_tc(q_local, k_full, v_full, do_local, lse_local, a.delta, dq_local,
                           dk_accum, dv_accum, d_meta, meta_bytes, (int)total_tokens, H, D,
                           (int)s_local, cp_size, rank, (int)strategy, softmax_scale,
                           softmax_scale * kLog2e, m, (int)operand_dtype, s);
}

extern "C" int cp_attn_bwd(const void* q_local, const void* k_full, const void* v_full,
                           const void* o_local, const void* o_resid_local,
                           const float* lse_local, const void* do_local,
                           void* dq_local, float* dk_accum, float* dv_accum, const void* d_meta,
                           size_t meta_bytes, int64_t total_tokens, int H, int D, int cp_size,
                           int rank, cp_strategy_t strategy, float softmax_scale,
                           cp_dtype_t operand_dtype, void* d_workspace, size_t workspace_bytes,
                           void* stream) {
  return cp_attn_bwd_ex(q_local, k_full, v_full, o_local, o_resid_local, lse_local, do_local,
                        dq_local, dk_accum,
                        dv_accum, d_meta, meta_bytes, total_tokens, H, D, cp_size, rank, strategy,
                        softmax_scale, operand_dtype, CP_BWD_ACCUMULATE, d_workspace,
                        workspace_bytes, stream);
}

extern "C" size_t cp_attn_bwd_grouped_workspace_bytes(int64_t s_local, int H, int cp_size,
                                                      int64_t total_tokens) {
  if (s_local < 0 || H < 1 || cp_size < 1 || total_tokens < 0) return 0;
  const size_t delta = (((size_t)cp_size * s_local * H * sizeof(float)) + 15) & ~(size_t)15;
  return delta + grouped_scratch_bytes(total_tokens);
}

static int bwd_grouped(const void* q_all, const void* k_full, const void* v_full,
                       const void* o_all, const void* o_resid_all, const float* lse_all,
                       const void* do_all, void* dq_all, float* dk_accum, float* dv_accum,
                       const void* d_meta_all, size_t meta_stride, int64_t total_tokens, int H,
                       int D, int cp_size, cp_strategy_t strategy, float softmax_scale,
                       cp_dtype_t operand_dtype, void* d_workspace, size_t workspace_bytes,
                       void* stream, void* dk_all, void* dv_all, const int32_t* d_restore) {
  if (check_dtype(operand_dtype) != CP_OK) return CP_ERR_INVALID_ARG;
  int64_t s_local = 0;
  int st = common_checks(q_all, k_full, v_full, d_meta_all, meta_stride, total_tokens, H, D,
                         cp_size, 0, strategy, &s_local);
  if (st != CP_OK) return st;
  if (meta_stride % 16) return CP_ERR_ALIGNMENT;
  const bool rs = dk_all != nullptr;  // the reduce-scatter's scatter fused in
  if (!o_all || !lse_all || !do_all || !dq_all || (rs ? !dv_all : (!dk_accum || !dv_accum)))
    return CP_ERR_INVALID_ARG;
  if (!cpthd_host::aligned16(o_all) || !cpthd_host::aligned16(lse_all) ||
      !cpthd_host::aligned16(do_all) || !cpthd_host::aligned16(dq_all) ||
      !cpthd_host::aligned16(dk_accum) || !cpthd_host::aligned16(dv_accum) ||
      !cpthd_host::aligned16(o_resid_all) || !cpthd_host::aligned16(dk_all) ||
      !cpthd_host::aligned16(dv_all))
    return CP_ERR_ALIGNMENT;
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return CP_ERR_INVALID_ARG;
  if (s_local == 0) return CP_OK;
  if (!d_workspace ||
      workspace_bytes < cp_attn_bwd_grouped_workspace_bytes(s_local, H, cp_size, total_tokens))
    return CP_ERR_WORKSPACE;
  if (!cpthd_host::aligned16(d_workspace)) return CP_ERR_ALIGNMENT;
  cudaStream_t s = cpthd_host::as_stream(stream);
  float* delta_all = (float*)d_workspace;
  void* scratch = (char*)d_workspace +
                  ((((size_t)cp_size * s_local * H * sizeof(float)) + 15) & ~(size_t)15);
  const size_t row_bytes = (size_t)H * D * 2;  // one row of a bf16 / fp16 [*, H, D] tensor
  // per rank: Delta, then dQ (the dK/dV of every rank follows in one launch)
  for (int r = 0; r < cp_size; ++r) {
    const size_t ro = (size_t)r * s_local * row_bytes;
    const void* meta_r = (const char*)d_meta_all + meta_stride * r;
    AttnArgs a{};
    a.out = (const bf16*)((const char*)o_all + ro);
    a.out_resid = o_resid_all ? (const bf16*)((const char*)o_resid_all + ro) : nullptr;
    a.dout = (const bf16*)((const char*)do_all + ro);
    a.delta = delta_all + (size_t)r * H * s_local;
    a.meta = meta_r; a.meta_bytes = meta_stride;
    a.T = (int)total_tokens; a.H = H; a.s_local = (int)s_local; a.cp = cp_size; a.rank = r;
    a.strategy = (int)strategy;
    if ((st = launch_delta(a, D, (int)operand_dtype, s)) != CP_OK) return st;
  }
  for (int r = 0; r < cp_size; ++r) {
    const size_t ro = (size_t)r * s_local * row_bytes;
    const void* meta_r = (const char*)d_meta_all + meta_stride * r;
    st = cpthd_attn_bwd_tc((const char*)q_all + ro, k_full, v_full, (const char*)do_all + ro,
                           lse_all + (size_t)r * H * s_local, delta_all + (size_t)r * H * s_local,
                           (char*)dq_all + ro, dk_accum, dv_accum, meta_r, meta_stride,
                           (int)total_tokens, H, D, (int)s_local, cp_size, r, (int)strategy,
                           softmax_scale, softmax_scale * kLog2e, kBwdDqOnly, (int)operand_dtype,
                           s, r > 0 ? 1 : 0);
    if (st != CP_OK) return st;
  }
  // the ranks' dQ launches after the first, the work-order kernel and the
  // dK/dV kernel each start as the previous grid drains (programmatic
  // dependent launch): none of them reads what the one before writes, except
  // the dK/dV kernel, which waits for the work order on the device
  return cpthd_attn_dkdv_grouped_tc(q_all, k_full, v_full, do_all, lse_all, delta_all, dk_accum,
                                    dv_accum, d_meta_all, meta_stride, (int)total_tokens, H, D,
                                    (int)s_local, cp_size, (int)strategy, softmax_scale,
                                    softmax_scale * kLog2e, (int)operand_dtype, scratch, s,
                                    dk_all, dv_all, d_restore, 2);
}

extern "C" int cp_attn_bwd_grouped(const void* q_all, const void* k_full, const void* v_full,
                                   const void* o_all, const void* o_resid_all,
                                   const float* lse_all, const void* do_all, void* dq_all,
                                   float* dk_accum, float* dv_accum, const void* d_meta_all,
                                   size_t meta_stride, int64_t total_tokens, int H, int D,
                                   int cp_size, cp_strategy_t strategy, float softmax_scale,
                                   cp_dtype_t operand_dtype, void* d_workspace,
                                   size_t workspace_bytes, void* stream) {
  return bwd_grouped(q_all, k_full, v_full, o_all, o_resid_all, lse_all, do_all, dq_all,
                     dk_accum, dv_accum, d_meta_all, meta_stride, total_tokens, H, D, cp_size,
                     strategy, softmax_scale, operand_dtype, d_workspace, workspace_bytes, stream,
                     nullptr, nullptr, nullptr);
}

extern "C" int cp_attn_bwd_grouped_rs(const void* q_all, const void* k_full, const void* v_full,
                                      const void* o_all, const void* o_resid_all,
                                      const float* lse_all, const void* do_all, void* dq_all,
                                      void* dk_all, void* dv_all, const int32_t* d_restore,
                                      const void* d_meta_all, size_t meta_stride,
                                      int64_t total_tokens, int H, int D, int cp_size,
                                      cp_strategy_t strategy, float softmax_scale,
                                      cp_dtype_t operand_dtype, void* d_workspace,
                                      size_t workspace_bytes, void* stream) {
  if (!dk_all || !dv_all) return CP_ERR_INVALID_ARG;
  if (strategy == CP_DUAL_CHUNK_SWAP && !d_restore) return CP_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(d_restore) & 3u) return CP_ERR_ALIGNMENT;
  return bwd_grouped(q_all, k_full, v_full, o_all, o_resid_all, lse_all, do_all, dq_all,
                     nullptr, nullptr, d_meta_all, meta_stride, total_tokens, H, D, cp_size,
                     strategy, softmax_scale, operand_dtype, d_workspace, workspace_bytes, stream,
                     dk_all, dv_all, d_restore);
}

extern "C" size_t cp_attn_bwd_ring_workspace_bytes(int64_t s_local, int H, int cp_size) {
  if (s_local < 0 || H < 1 || cp_size < 1) return 0;
  const size_t delta = (((size_t)cp_size * s_local * H * sizeof(float)) + 15) & ~(size_t)15;
  return delta + ring_bwd_scratch_bytes(s_local, cp_size);
}

static int bwd_ring(const void* q_all, const void* k_shards, const void* v_shards,
                    const void* o_all, const void* o_resid_all, const float* lse_all,
                    const void* do_all, void* dq_all, float* dk_accum, float* dv_accum,
                    const void* d_ring_meta, size_t step_bytes, size_t rank_stride, int64_t s_local,
                    int H, int D, int cp_size, cp_strategy_t strategy, float softmax_scale,
                    cp_dtype_t operand_dtype, void* d_workspace, size_t workspace_bytes,
                    void* stream, void* dk_all, void* dv_all) {
  if (check_dtype(operand_dtype) != CP_OK) return CP_ERR_INVALID_ARG;
  const bool rs = dk_all != nullptr;  // bf16 dK / dV out, the cast fused in
  if (!q_all || !k_shards || !v_shards || !o_all || !lse_all || !do_all || !dq_all ||
      (rs ? !dv_all : (!dk_accum || !dv_accum)) || !d_ring_meta)
    return CP_ERR_INVALID_ARG;
  if (H < 1 || cp_size < 1 || s_local < 0 || s_local * cp_size > INT32_MAX)
    return CP_ERR_INVALID_ARG;
  if (strategy != CP_DUAL_CHUNK_SWAP && strategy != CP_NO_LOAD_BALANCE) return CP_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return CP_ERR_UNSUPPORTED;
  if (H > 65535 || (int64_t)s_local * cp_size * H * D > ((int64_t)1 << 40)) return CP_ERR_UNSUPPORTED;
  // a shard's last key block may hold fewer than 128 rows; its 32-row output
  // chunks must not reach into the next shard's rows
  if (s_local % 32) return CP_ERR_UNSUPPORTED;
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return CP_ERR_INVALID_ARG;
  if (step_bytes < 64 || rank_stride < step_bytes * (size_t)cp_size) return CP_ERR_WORKSPACE;
  if (step_bytes % 16 || rank_stride % 16) return CP_ERR_ALIGNMENT;
  if (!cpthd_host::aligned16(q_all) || !cpthd_host::aligned16(k_shards) ||
      !cpthd_host::aligned16(v_shards) || !cpthd_host::aligned16(o_all) ||
      !cpthd_host::aligned16(o_resid_all) || !cpthd_host::aligned16(lse_all) ||
      !cpthd_host::aligned16(do_all) || !cpthd_host::aligned16(dq_all) ||
      !cpthd_host::aligned16(dk_accum) || !cpthd_host::aligned16(dv_accum) ||
      !cpthd_host::aligned16(d_ring_meta) || !cpthd_host::aligned16(dk_all) ||
      !cpthd_host::aligned16(dv_all))
    return CP_ERR_ALIGNMENT;
  if (s_local == 0) return CP_OK;
  if (!d_workspace || workspace_bytes < cp_attn_bwd_ring_workspace_bytes(s_local, H, cp_size))
    return CP_ERR_WORKSPACE;
  if (!cpthd_host::aligned16(d_workspace)) return CP_ERR_ALIGNMENT;
  cudaStream_t s = cpthd_host::as_stream(stream);
  float* delta_all = (float*)d_workspace;
  void* scratch = (char*)d_workspace +
                  ((((size_t)cp_size * s_local * H * sizeof(float)) + 15) & ~(size_t)15);
  const size_t row_bytes = (size_t)H * D * 2;
  int st;
  for (int r = 0; r < cp_size; ++r) {  // Delta of every rank, once (not once per ring step)
    const size_t ro = (size_t)r * s_local * row_bytes;
    AttnArgs a{};
    a.out = (const bf16*)((const char*)o_all + ro);
    a.out_resid = o_resid_all ? (const bf16*)((const char*)o_resid_all + ro) : nullptr;
    a.dout = (const bf16*)((const char*)do_all + ro);
    a.delta = delta_all + (size_t)r * H * s_local;
    a.H = H; a.s_local = (int)s_local;
    if ((st = launch_delta(a, D, (int)operand_dtype, s)) != CP_OK) return st;
  }
  return cpthd_attn_bwd_ring_tc(q_all, k_shards, v_shards, do_all, lse_all, delta_all, dq_all,
                                dk_accum, dv_accum, d_ring_meta, step_bytes, rank_stride, H, D,
                                (int)s_local, cp_size, (int)strategy, softmax_scale,
                                softmax_scale * kLog2e, (int)operand_dtype, scratch, s, dk_all,
                                dv_all);
}

extern "C" int cp_attn_bwd_ring(const void* q_all, const void* k_shards, const void* v_shards,
                                const void* o_all, const void* o_resid_all, const float* lse_all,
                                const void* do_all, void* dq_all, float* dk_accum, float* dv_accum,
                                const void* d_ring_meta, size_t step_bytes, size_t rank_stride,
                                int64_t s_local, int H, int D, int cp_size,
                                cp_strategy_t strategy, float softmax_scale,
                                cp_dtype_t operand_dtype, void* d_workspace,
                                size_t workspace_bytes, void* stream) {
  return bwd_ring(q_all, k_shards, v_shards, o_all, o_resid_all, lse_all, do_all, dq_all,
                  dk_accum, dv_accum, d_ring_meta, step_bytes, rank_stride, s_local, H, D, cp_size,
                  strategy, softmax_scale, operand_dtype, d_workspace, workspace_bytes, stream,
                  nullptr, nullptr);
}

extern "C" int cp_attn_bwd_ring_rs(const void* q_all, const void* k_shards, const void* v_shards,
                                   const void* o_all, const void* o_resid_all,
                                   const float* lse_all, const void* do_all, void* dq_all,
                                   void* dk_all, void* dv_all, const void* d_ring_meta,
                                   size_t step_bytes, size_t rank_stride, int64_t s_local, int H,
                                   int D, int cp_size, cp_strategy_t strategy,
                                   float softmax_scale, cp_dtype_t operand_dtype,
                                   void* d_workspace, size_t workspace_bytes, void* stream) {
  if (!dk_all || !dv_all) return CP_ERR_INVALID_ARG;
  return bwd_ring(q_all, k_shards, v_shards, o_all, o_resid_all, lse_all, do_all, dq_all, nullptr,
                  nullptr, d_ring_meta, step_bytes, rank_stride, s_local, H, D, cp_size, strategy,
                  softmax_scale, operand_dtype, d_workspace, workspace_bytes, stream, dk_all,
                  dv_all);
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
unsigned long long g_noalloc_ctx[kMaxDevices] = {};  // context the address belongs to

// Unique id of the calling thread's current CUDA context (0 when none is
// current or the driver cannot say).  A cudaDeviceReset ends the primary
// context; the one that replaces it has a new id.
unsigned long long current_context_id() {
  static std::once_flag once;
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_noalloc_scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// with the device current, once per device and context, and kept: a new
// context on the device (after a cudaDeviceReset) has the module loaded anew,
// so the address is looked up again.  Without a context id the lookup is
// repeated on every call.
int noalloc_scratch(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CP_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return CP_ERR_UNSUPPORTED;
  const unsigned long long id = current_context_id();
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev] || id == 0 || id != g_noalloc_ctx[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return CP_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<float*>(p);
    // the lookup made the device's primary context current if none was
    g_noalloc_ctx[dev] = id != 0 ? id : current_context_id();
  }
  *out = g_noalloc_ptr[dev];
  return CP_OK;
}

}  // namespace

extern "C" int cp_attn_bwd_noalloc(const void* q_local, const void* k_full, const void* v_full,
                                   const void* o_local, const void* o_resid_local,
                                   const float* lse_local,
                                   const void* do_local, void* dq_local, float* dk_accum,
                                   float* dv_accum, const void* d_meta, size_t meta_bytes,
                                   int64_t total_tokens, int H, int D, int cp_size, int rank,
                                   cp_strategy_t strategy, float softmax_scale,
                                   cp_dtype_t operand_dtype, void* stream) {
  int64_t s_local = 0;
  int st = common_checks(q_local, k_full, v_full, d_meta, meta_bytes, total_tokens, H, D, cp_size,
                         rank, strategy, &s_local);
  if (st != CP_OK) return st;
  if (!o_local || !lse_local || !do_local || !dq_local || !dk_accum || !dv_accum)
    return CP_ERR_INVALID_ARG;
  if (!cpthd_host::aligned16(o_local) || !cpthd_host::aligned16(lse_local) ||
      !cpthd_host::aligned16(do_local) || !cpthd_host::aligned16(dq_local) ||
      !cpthd_host::aligned16(dk_accum) || !cpthd_host::aligned16(dv_accum) ||
      !cpthd_host::aligned16(o_resid_local))
    return CP_ERR_ALIGNMENT;
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return CP_ERR_INVALID_ARG;
  if ((st = check_dtype(operand_dtype)) != CP_OK) return st;
  if (s_local * (int64_t)H > (int64_t)CP_NOALLOC_MAX_SCRATCH_FLOATS) return CP_ERR_WORKSPACE;
  if (s_local == 0) return CP_OK;
  float* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != CP_OK) return st;
  AttnArgs a{};
  a.q = (const bf16*)q_local; a.k = (const bf16*)k_full; a.v = (const bf16*)v_full;
  a.out = (const bf16*)o_local; a.out_resid = (const bf16*)o_resid_local;
  a.lse = const_cast<float*>(lse_local);
  a.dout = (const bf16*)do_local; a.dq = (bf16*)dq_local; a.dk = dk_accum; a.dv = dv_accum;
  a.delta = scratch; a.meta = d_meta; a.meta_bytes = meta_bytes;
  a.T = (int)total_tokens; a.H = H; a.s_local = (int)s_local; a.cp = cp_size; a.rank = rank;
  a.strategy = (int)strategy; a.scale = softmax_scale; a.scale_log2 = softmax_scale * kLog2e;
  cudaStream_t s = cpthd_host::as_stream(stream);
  if ((st = launch_delta(a, D, (int)operand_dtype, s)) != CP_OK) return st;
  return cpthd_attn_bwd_tc(q_local, k_full, v_full, do_local, lse_local, a.delta, dq_local,
                           dk_accum, dv_accum, d_meta, meta_bytes, (int)total_tokens, H, D,
                           (int)s_local, cp_size, rank, (int)strategy, softmax_scale,
                           softmax_scale * kLog2e, 0, (int)operand_dtype, s);
}
