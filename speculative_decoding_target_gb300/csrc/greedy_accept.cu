// Greedy acceptance: per-row vocabulary argmax, then the accepted prefix
// and the bonus token per request ("DFlash to dLLM self-spec, part 1",
// section 1.1 verify comparison table, section 1.3.3 accept/bonus kernel,
// section 1.6.1 commit_lens = accept_len + 1).
//
// Kernel 1 streams the fp32 logits once: CTA (chunk, row) reduces 8192
// entries with 16-byte streaming loads to a (value, index) pair.  Kernel 2,
// one CTA per request, reduces the chunk pairs of its q_len rows and walks
// the drafts.  The reduction order is arbitrary, so the combine is a total
// order that makes the result unique: NaN above every number (lower index
// first among NaNs), then larger value, then lower index (so -0 == +0 ties
// go to the lower index).
#include <climits>

#include "common.cuh"

namespace specv {
namespace {

__device__ __forceinline__ bool better(float a, int ia, float b, int ib) {
  const bool na = a != a, nb = b != b;
  if (na || nb) return na && (!nb || ia < ib);
  return a > b || (a == b && ia < ib);
}

__device__ __forceinline__ void take(float v, int i, float& bv, int& bi) {
  if (better(v, i, bv, bi)) {
    bv = v;
    bi = i;
  }
}

__device__ __forceinline__ void warp_argmax(float& bv, int& bi) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    take(ov, oi, bv, bi);
  }
}

__global__ void __launch_bounds__(kAcceptThreads)
    argmax_partial_kernel(const AcceptParams p) {
  const int chunk = blockIdx.x, row = blockIdx.y;
  const float* x = p.logits + (long long)row * p.vocab;
  const int begin = chunk * kAcceptChunk;
  const int end = min(begin + kAcceptChunk, p.vocab);
  float bv = -INFINITY;
  int bi = INT_MAX;
  if (p.vec4) {
    // 8192 floats = 2048 float4 = 8 per thread, all loads issued first
    const float4* x4 = reinterpret_cast<const float4*>(x + begin);
    const int n4 = (end - begin) >> 2;
    float4 v[kAcceptChunk / 4 / kAcceptThreads];
#pragma unroll
    for (int k = 0; k < kAcceptChunk / 4 / kAcceptThreads; ++k) {
      const int j = threadIdx.x + k * kAcceptThreads;
      v[k] = j < n4 ? __ldcs(x4 + j)
                    : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
#pragma unroll
    for (int k = 0; k < kAcceptChunk / 4 / kAcceptThreads; ++k) {
      const int j = threadIdx.x + k * kAcceptThreads;
      if (j < n4) {
        const int i0 = begin + 4 * j;
        take(v[k].x, i0, bv, bi);
        take(v[k].y, i0 + 1, bv, bi);
        take(v[k].z, i0 + 2, bv, bi);
        take(v[k].w, i0 + 3, bv, bi);
      }
    }
  } else {
    for (int i = begin + threadIdx.x; i < end; i += kAcceptThreads)
      take(__ldcs(x + i), i, bv, bi);
  }
  warp_argmax(bv, bi);
  __shared__ float s_v[kAcceptThreads / 32];
  __shared__ int s_i[kAcceptThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    s_v[warp] = bv;
    s_i[warp] = bi;
  }
  __syncthreads();
  if (warp == 0) {
    bv = lane < kAcceptThreads / 32 ? s_v[lane] : -INFINITY;
    bi = lane < kAcceptThreads / 32 ? s_i[lane] : INT_MAX;
    warp_argmax(bv, bi);
    if (lane == 0) {
      p.part_val[(long long)row * p.chunks + chunk] = bv;
      p.part_idx[(long long)row * p.chunks + chunk] = bi;
    }
  }
}

__global__ void accept_finalize_kernel(const AcceptParams p) {
  __shared__ int s_t[32];
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp < p.q_len) {
    const long long row = (long long)b * p.q_len + warp;
    float bv = -INFINITY;
    int bi = INT_MAX;
    for (int c = lane; c < p.chunks; c += 32)
      take(p.part_val[row * p.chunks + c], p.part_idx[row * p.chunks + c], bv,
           bi);
    warp_argmax(bv, bi);
    if (lane == 0) s_t[warp] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int32_t* d = p.draft_ids + (long long)b * p.q_len;
    int a = 0;
    while (a + 1 < p.q_len && d[a + 1] == s_t[a]) ++a;
    p.accept_len[b] = a;
    p.next_token[b] = s_t[a];
    if (p.out_tokens) {
      int32_t* o = p.out_tokens + (long long)b * p.q_len;
      for (int j = 0; j < p.q_len; ++j)
        o[j] = j < a ? d[j + 1] : (j == a ? s_t[a] : -1);
    }
  }
}

}  // namespace

cudaError_t launch_greedy_accept(const AcceptParams& p, cudaStream_t s) {
  dim3 g1(p.chunks, p.rows);
  argmax_partial_kernel<<<g1, kAcceptThreads, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  accept_finalize_kernel<<<p.batch, 32 * p.q_len, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace specv
