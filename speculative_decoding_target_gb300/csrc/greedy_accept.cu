// Greedy acceptance: per-row vocabulary argmax, then the accepted prefix
// and the bonus token per request ("DFlash to dLLM self-spec, part 1",
// section 1.1 verify comparison table, section 1.3.3 accept/bonus kernel,
// section 1.6.1 commit_lens = accept_len + 1).
//
// One launch streams the fp32 logits once: CTA (chunk, row) reduces 8192
// entries with 16-byte streaming loads to a (maximum, first index) pair;
// rows past a request's block width are skipped unread.  The last CTA of a
// request to finish (a per-request counter, zeroed before the launch) then
// reduces the chunk pairs of its rows, walks the drafts and publishes the
// committed cache length.  The reduction order is arbitrary, so the combine is a total
// order that makes the result unique: NaN above every number (lower index
// first among NaNs), then larger value, then lower index (so -0 == +0 ties
// go to the lower index).
#include <climits>

#include "accept.cuh"
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

// Maximum that propagates NaN (IEEE maxNum would drop it).
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

__device__ __forceinline__ bool hits(float e, float M, bool nanM) {
  return nanM ? e != e : e == M;
}

// The chunk pair of (chunk, row), by one CTA.  Pass 1 takes the chunk's
// maximum with one NaN-propagating max per logit; only threads that hold
// that maximum then look for its first index among their own logits (in
// index order), and the smallest such index wins.  The pair (maximum, first
// index) is the same one the total order above selects.
__device__ __forceinline__ void chunk_argmax(const AcceptParams& p, int chunk,
                                             int row) {
  constexpr int kVec = kAcceptChunk / 4 / kAcceptThreads;  // float4 per thread
  __shared__ float s_m[kAcceptThreads / 32];
  __shared__ int s_i[kAcceptThreads / 32];
  const float* x = p.logits + (long long)row * p.vocab;
  const int begin = chunk * kAcceptChunk;
  const int end = min(begin + kAcceptChunk, p.vocab);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float m = -INFINITY;
  float4 v[kVec];
  const int n4 = (end - begin) >> 2;
  if (p.vec4) {
    const float4* x4 = reinterpret_cast<const float4*>(x + begin);
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int j = threadIdx.x + k * kAcceptThreads;
      v[k] = j < n4 ? __ldcs(x4 + j)
                    : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
#pragma unroll
    for (int k = 0; k < kVec; ++k)
      m = max_nan(max_nan(max_nan(m, v[k].x), max_nan(v[k].y, v[k].z)), v[k].w);
  } else {
    for (int i = begin + threadIdx.x; i < end; i += kAcceptThreads)
      m = max_nan(m, __ldcs(x + i));
  }
  // chunk maximum
  float M = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    M = max_nan(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (lane == 0) s_m[warp] = M;
  __syncthreads();
  M = s_m[0];
#pragma unroll
  for (int w = 1; w < kAcceptThreads / 32; ++w) M = max_nan(M, s_m[w]);
  const bool nanM = M != M;
  // first index of the maximum among this thread's logits
  int cand = INT_MAX;
  if (hits(m, M, nanM)) {
    if (p.vec4) {
#pragma unroll
      for (int k = 0; k < kVec; ++k) {
        const int j = threadIdx.x + k * kAcceptThreads;
        const int i0 = begin + 4 * j;
        if (j < n4 && cand == INT_MAX) {
          if (hits(v[k].x, M, nanM)) cand = i0;
          else if (hits(v[k].y, M, nanM)) cand = i0 + 1;
          else if (hits(v[k].z, M, nanM)) cand = i0 + 2;
          else if (hits(v[k].w, M, nanM)) cand = i0 + 3;
        }
      }
    } else {
      for (int i = begin + threadIdx.x; i < end; i += kAcceptThreads)
        if (hits(x[i], M, nanM)) {
          cand = i;
          break;
        }
    }
  }
  cand = __reduce_min_sync(0xffffffffu, cand);
  if (lane == 0) s_i[warp] = cand;
  __syncthreads();
  if (threadIdx.x == 0) {
    int best = s_i[0];
#pragma unroll
    for (int w = 1; w < kAcceptThreads / 32; ++w) best = min(best, s_i[w]);
    p.part_val[(long long)row * p.chunks + chunk] = M;
    p.part_idx[(long long)row * p.chunks + chunk] = best;
  }
}

// Request b's accepted prefix and bonus token from its rows' chunk pairs,
// by one CTA (the pairs are read past L1: other CTAs wrote them).
__device__ __forceinline__ void finalize_request(const AcceptParams& p, int b) {
  __shared__ int s_t[16], s_d[16];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qb = p.q_lens ? min(max(p.q_lens[b], 0), p.q_len) : p.q_len;
  // the drafts, loaded side by side rather than one by one in the walk
  if (threadIdx.x < p.q_len)
    s_d[threadIdx.x] = p.draft_ids[(long long)b * p.q_len + threadIdx.x];
  for (int j = warp; j < qb; j += kAcceptThreads / 32) {
    const long long row = (long long)b * p.q_len + j;
    float bv = -INFINITY;
    int bi = INT_MAX;
    for (int c = lane; c < p.chunks; c += 32)
      take(__ldcg(p.part_val + row * p.chunks + c),
           __ldcg(p.part_idx + row * p.chunks + c), bv, bi);
    warp_argmax(bv, bi);
    if (lane == 0) s_t[j] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int* d = s_d;
    int a = 0;
    while (a + 1 < qb && d[a + 1] == s_t[a]) ++a;
    // an idle request (no rows) commits nothing
    const int next = qb > 0 ? s_t[a] : -1;
    p.accept_len[b] = a;
    p.next_token[b] = next;
    if (p.out_tokens) {
      int32_t* o = p.out_tokens + (long long)b * p.q_len;
      for (int j = 0; j < p.q_len; ++j)
        o[j] = j < a ? d[j + 1] : (j == a ? next : -1);
    }
    // the cache keeps the prefix, the boundary and d1..da
    if (p.new_seq_lens)
      p.new_seq_lens[b] = qb > 0 ? p.seq_lens[b] - qb + a + 1 : p.seq_lens[b];
  }
}

// CTA (chunk, row): the chunk pair, then the per-request count; the
// request's last CTA to finish reduces its rows.
__global__ void __launch_bounds__(kAcceptThreads)
    argmax_partial_kernel(const AcceptParams p) {
  // a following attention call may be scheduled now (it waits for this
  // grid before touching memory)
  tc_grid_launch_dependents();
  const int chunk = blockIdx.x, row = blockIdx.y;
  const int b = row / p.q_len;
  // uniform per CTA: a row past its block is not read, only counted
  if (!p.q_lens || row - b * p.q_len < min(max(p.q_lens[b], 0), p.q_len))
    chunk_argmax(p, chunk, row);
  __shared__ int s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    // thread 0 wrote this CTA's pair: a release add orders it before the
    // count, and the acquire side makes every counted pair visible to the
    // last CTA (its other threads through the barrier below)
    int old;
    asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;"
                 : "=r"(old)
                 : "l"(p.counters + b)
                 : "memory");
    s_last = old == p.q_len * p.chunks - 1;
  }
  __syncthreads();
  if (s_last) finalize_request(p, b);
}

}  // namespace

cudaError_t launch_greedy_accept(const AcceptParams& p, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(p.counters, 0, sizeof(int32_t) * p.batch, s);
  if (e != cudaSuccess) return e;
  dim3 g1(p.chunks, p.rows);
  argmax_partial_kernel<<<g1, kAcceptThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace specv
