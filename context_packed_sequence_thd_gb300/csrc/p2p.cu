// p2p.cu -- merge of the per-step partial attention outputs of the ring
// (P2P) comm type ("THD P2P context-parallel regression when padded
// cu_seqlens are value-equal but not object-identical", §Describe the bug:
// the P2P context-parallel path), every rank on one GPU.
//
// At ring step i a rank's queries attend one K/V shard only, giving a
// partial output O_i (bf16, normalised over that shard's keys) and its
// log-sum-exp LSE_i (-inf where a row saw no key of the shard).  Attention
// over the union of the shards is the softmax-weighted combination
//   LSE = log sum_i exp(LSE_i),   O = sum_i exp(LSE_i - LSE) * O_i,
// computed here in fp32 and rounded to bf16 once.  With the steps' rounding
// remainders (O_i's bf16 remainder, as the attention forward writes it) the
// sum reads O_i to about 16 bits, and the merged output's own remainder can
// be written too, for the backward's Delta.
//
// Design: bandwidth bound (n_steps + 1 rows of 2*H*D bytes per (row, head)
// pair moved, a few flops per byte).  One thread owns 8 columns (16 bytes)
// of one (row, head) pair; consecutive threads cover consecutive 16-byte
// chunks of the [s_local, H, D] rows, so every step's loads and the store are
// fully coalesced.  Steps whose weight is zero (no key seen) are not read.
// Grid: a multiple of the SM count, grid-stride loop.
#include "common.cuh"

namespace cpthd {
namespace {

constexpr int kMergeThreads = 256;

__device__ __forceinline__ uint4 ld_once(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <int D>
__global__ void __launch_bounds__(kMergeThreads)
p2p_merge_kernel(const uint4* __restrict__ o_steps, const uint4* __restrict__ o_steps_resid,
                 const float* __restrict__ lse_steps, int n_steps, int64_t s_local, int H,
                 uint4* __restrict__ out, uint4* __restrict__ out_resid,
                 float* __restrict__ lse_out) {
  constexpr int G = D / 8;  // threads per (row, head) pair
  const int64_t n_pairs = s_local * H;
  const int64_t n_chunks = n_pairs * G;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_chunks;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t pair = i / G;
    const int64_t row = pair / H;
    const int h = (int)(pair - row * H);
    const int64_t li = (int64_t)h * s_local + row;  // [H, s_local] position
    float m = -INFINITY;
    for (int s = 0; s < n_steps; ++s) m = fmaxf(m, lse_steps[s * n_pairs + li]);
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    float lse = -INFINITY;
    if (m != -INFINITY) {
      float sum = 0.f;
      for (int s = 0; s < n_steps; ++s) sum += expf(lse_steps[s * n_pairs + li] - m);
      lse = m + logf(sum);
#pragma unroll 4
      for (int s = 0; s < n_steps; ++s) {
        const float l = lse_steps[s * n_pairs + li];
        if (l == -INFINITY) continue;
        const float w = expf(l - lse);
        const uint4 x = ld_once(o_steps + s * n_chunks + i);
        const uint4 xr = o_steps_resid ? ld_once(o_steps_resid + s * n_chunks + i)
                                       : make_uint4(0, 0, 0, 0);
        const __nv_bfloat162* xp = reinterpret_cast<const __nv_bfloat162*>(&x);
        const __nv_bfloat162* rp = reinterpret_cast<const __nv_bfloat162*>(&xr);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(xp[e]), fr = __bfloat1622float2(rp[e]);
          acc[2 * e] = fmaf(w, f.x + fr.x, acc[2 * e]);
          acc[2 * e + 1] = fmaf(w, f.y + fr.y, acc[2 * e + 1]);
        }
      }
    }
    uint4 r;
    r.x = pack_bf16(acc[0], acc[1]);
    r.y = pack_bf16(acc[2], acc[3]);
    r.z = pack_bf16(acc[4], acc[5]);
    r.w = pack_bf16(acc[6], acc[7]);
    out[i] = r;
    if (out_resid) {
      uint4 q;
      q.x = pack_bf16(acc[0] - bf16_lo_f(r.x), acc[1] - bf16_hi_f(r.x));
      q.y = pack_bf16(acc[2] - bf16_lo_f(r.y), acc[3] - bf16_hi_f(r.y));
      q.z = pack_bf16(acc[4] - bf16_lo_f(r.z), acc[5] - bf16_hi_f(r.z));
      q.w = pack_bf16(acc[6] - bf16_lo_f(r.w), acc[7] - bf16_hi_f(r.w));
      out_resid[i] = q;
    }
    if (i % G == 0) lse_out[li] = lse;
  }
}

}  // namespace
}  // namespace cpthd

using namespace cpthd;

extern "C" int cp_p2p_merge(const void* d_o_steps, const void* d_o_steps_resid,
                            const float* d_lse_steps, int n_steps, int64_t s_local, int H, int D,
                            void* d_out, void* d_out_resid, float* d_lse, void* stream) {
  if (!d_o_steps || !d_lse_steps || !d_out || !d_lse) return CP_ERR_INVALID_ARG;
  if (n_steps < 1 || s_local < 0 || H < 1) return CP_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return CP_ERR_UNSUPPORTED;
  if (s_local * H * (int64_t)D * n_steps > ((int64_t)1 << 40)) return CP_ERR_UNSUPPORTED;
  if (!cpthd_host::aligned16(d_o_steps) || !cpthd_host::aligned16(d_lse_steps) ||
      !cpthd_host::aligned16(d_out) || !cpthd_host::aligned16(d_lse) ||
      !cpthd_host::aligned16(d_o_steps_resid) || !cpthd_host::aligned16(d_out_resid))
    return CP_ERR_ALIGNMENT;
  if (s_local == 0) return CP_OK;
  const int64_t chunks = s_local * H * (D / 8);
  const int64_t want = (chunks + kMergeThreads - 1) / kMergeThreads;
  const int sms = cpthd_host::sm_count();
  const int grid = (int)std::min<int64_t>(want, (int64_t)sms * 8);
  cudaStream_t s = cpthd_host::as_stream(stream);
  const uint4* o = reinterpret_cast<const uint4*>(d_o_steps);
  const uint4* o_r = reinterpret_cast<const uint4*>(d_o_steps_resid);
  uint4* out = reinterpret_cast<uint4*>(d_out);
  uint4* out_r = reinterpret_cast<uint4*>(d_out_resid);
  if (D == 64)
    p2p_merge_kernel<64><<<grid, kMergeThreads, 0, s>>>(o, o_r, d_lse_steps, n_steps, s_local, H,
                                                        out, out_r, d_lse);
  else
    p2p_merge_kernel<128><<<grid, kMergeThreads, 0, s>>>(o, o_r, d_lse_steps, n_steps, s_local, H,
                                                         out, out_r, d_lse);
  return cpthd_host::launch_status();
}
