// Block KV append with FP8 quantise-on-write, plus the block's positions and
// cache locations.
//
// One warp per (request b, block row i, KV head g); lane l owns channels
// 8l .. 8l+7 (16 bytes of the bf16 input row).  For an FP8 pool the eight
// lanes of a 64-channel block reduce |x| by shuffles; the scale and the
// codes are computed in fp32 with correctly rounded division, so the stored
// bytes follow the rule stated in spec_verify.h exactly:
//   scale = fp16_rn(amax / 448) (1 if it rounds to zero),
//   byte  = E4M3_rn_satfinite(x / scale)
// ("Qwen3.8-27B-FP8" page, "Implemented execution path": E4M3 cache with
// per-token / per-KV-head FP16 scales over 64-channel blocks).
#include <cuda_fp8.h>

#include "append.cuh"
#include "common.cuh"
#include "spec_verify.h"

namespace specv {
namespace {

constexpr int kWarps = 4;

__global__ void __launch_bounds__(kWarps * 32)
    kv_append_kernel(const AppendParams p) {
  // the attention call that follows may be scheduled now (it waits for
  // this grid before touching memory)
  specv::tc_grid_launch_dependents();
  const int w = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (w >= p.batch * p.q_len * p.hkv) return;  // uniform per warp
  const int g = w % p.hkv;
  const int bi = w / p.hkv;
  const int i = bi % p.q_len, b = bi / p.q_len;
  int qb = p.q_len;
  if (p.q_lens) qb = min(max(p.q_lens[b], 0), p.q_len);
  const long long t = (long long)p.seq_lens[b] - qb + i;
  long long loc = -1;
  int page = 0;
  if (i < qb && t >= 0 && t < p.max_tokens) {
    page = p.page_table[(long long)b * p.max_pages + (t >> p.log2_ps)];
    if (page >= 0 && page < p.num_pages) {
      loc = (long long)page * p.page_size + (t & (p.page_size - 1));
    } else if (p.status && lane == 0) {
      atomicOr(p.status, SPEC_STATUS_BAD_PAGE);
    }
  }
  if (g == 0 && lane == 0) {
    if (p.positions) p.positions[bi] = i < qb && t >= 0 ? (int32_t)t : -1;
    if (p.cache_loc) p.cache_loc[bi] = loc;
  }
  if (loc < 0) return;
  const long long row = ((long long)page * p.hkv + g) * p.page_size +
                        (t & (p.page_size - 1));
  const long long src = (((long long)b * p.q_len + i) * p.hkv + g) * kHeadDim;
#pragma unroll
  for (int kv = 0; kv < 2; ++kv) {
    const __nv_bfloat16* in = kv ? p.v_new : p.k_new;
    const uint4 raw = *reinterpret_cast<const uint4*>(in + src + lane * 8);
    if (!p.fp8) {
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(kv ? p.v_pages : p.k_pages);
      *reinterpret_cast<uint4*>(dst + row * kHeadDim + lane * 8) = raw;
      continue;
    }
    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
    float x[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[2 * e] = __low2float(h2[e]);
      x[2 * e + 1] = __high2float(h2[e]);
    }
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1)  // the 8 lanes of this 64-channel block
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    __half scale = __float2half_rn(__fdiv_rn(amax, 448.f));
    if (__half2float(scale) == 0.f) scale = __float2half_rn(1.f);
    const float sf = __half2float(scale);
    uint32_t packed[2] = {0u, 0u};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 qv = make_float2(__fdiv_rn(x[2 * e], sf),
                                    __fdiv_rn(x[2 * e + 1], sf));
      const uint32_t pair =
          __nv_cvt_float2_to_fp8x2(qv, __NV_SATFINITE, __NV_E4M3) & 0xFFFFu;
      packed[e >> 1] |= pair << (16 * (e & 1));
    }
    uint8_t* dst = static_cast<uint8_t*>(kv ? p.v_pages : p.k_pages);
    *reinterpret_cast<uint2*>(dst + row * kHeadDim + lane * 8) =
        make_uint2(packed[0], packed[1]);
    if ((lane & 7) == 0) {
      __half* sdst = kv ? p.v_scales : p.k_scales;
      sdst[row * (kHeadDim / 64) + (lane >> 3)] = scale;
    }
  }
}

}  // namespace

cudaError_t launch_kv_append(const AppendParams& p, cudaStream_t s) {
  const int warps = p.batch * p.q_len * p.hkv;
  if (warps == 0) return cudaSuccess;
  kv_append_kernel<<<(warps + kWarps - 1) / kWarps, kWarps * 32, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace specv
