// Stochastic verify: speculative sampling against target and draft
// probabilities ("MTP and DFlash2 at long context on XPU", Part II: sampling
// needs rejection sampling against target and draft probabilities; the rule
// is that of Leviathan et al. 2023 and Chen et al. 2023).  p_j is the
// softmax of logits row j at the request's temperature; draft j is accepted
// iff u_j * q_j(d_j) < p_{j-1}(d_j); the first rejection draws the next
// token from max(0, p_{j-1} - q_j), full acceptance from p_{q_b-1}.  A
// draw from weights w with the uniform u is the smallest index whose running
// sum exceeds u * sum(w).
//
// Three launches:
//   1. softmax_partial_kernel, CTA (chunk, row): the chunk's maximum M and
//      sum exp2((x - M) k), k = log2(e) / T, in one streaming pass over the
//      logits (rows past a request's width are skipped unread);
//   2. residual_chunk_kernel, CTA (chunk, request): the accept walk (cheap,
//      repeated by every CTA of the request), then the chunk's total draw
//      weight;
//   3. sample_finalize_kernel, one CTA per request: the walk again, the
//      chunk that holds u * W, and a block scan of that chunk alone.
// Every float step that decides an integer goes through the same device
// functions in kernels 2 and 3 with explicitly rounded operations, so both
// see bit-identical weights.
#include <climits>

#include "stochastic.cuh"

namespace specv {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ int rows_of(const StochasticParams& p, int b) {
  return p.q_lens ? min(max(p.q_lens[b], 0), p.q_len) : p.q_len;
}

__device__ __forceinline__ float k_of(const StochasticParams& p, int b) {
  return __fdiv_rn(kLog2e, p.temperature[b]);
}

__device__ __forceinline__ float block_sum(float v, float* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s = __fadd_rn(s, red[w]);
  return s;
}

__global__ void __launch_bounds__(kSampleThreads)
    softmax_partial_kernel(const StochasticParams p) {
  constexpr int kVec = kSampleChunk / 4 / kSampleThreads;
  __shared__ float red[kSampleThreads / 32];
  const int chunk = blockIdx.x, row = blockIdx.y;
  const int b = row / p.q_len;
  if (row - b * p.q_len >= rows_of(p, b)) return;  // uniform per CTA
  const float k = k_of(p, b);
  const float* x = p.logits + (long long)row * p.vocab;
  const int begin = chunk * kSampleChunk;
  const int end = min(begin + kSampleChunk, p.vocab);
  float v[4 * kVec];  // entries past the row's end read as -inf
  if (p.vec4) {
    const float4* x4 = reinterpret_cast<const float4*>(x + begin);
    const int n4 = (end - begin) >> 2;
#pragma unroll
    for (int e = 0; e < kVec; ++e) {
      const int j = threadIdx.x + e * kSampleThreads;
      const float4 t = j < n4 ? __ldcs(x4 + j)
                              : make_float4(-INFINITY, -INFINITY, -INFINITY,
                                            -INFINITY);
      v[4 * e] = t.x; v[4 * e + 1] = t.y; v[4 * e + 2] = t.z; v[4 * e + 3] = t.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 4 * kVec; ++e) {
      const int i = begin + threadIdx.x + e * kSampleThreads;
      v[e] = i < end ? __ldcs(x + i) : -INFINITY;
    }
  }
  float m = -INFINITY;
#pragma unroll
  for (int e = 0; e < 4 * kVec; ++e) m = fmaxf(m, v[e]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = m;
  __syncthreads();
  float M = red[0];
  for (int w = 1; w < kSampleThreads / 32; ++w) M = fmaxf(M, red[w]);
  float s = 0.f;
  if (M != -INFINITY) {
#pragma unroll
    for (int e = 0; e < 4 * kVec; ++e) s += exp2f((v[e] - M) * k);
  }
  const float S = block_sum(s, red);
  if (threadIdx.x == 0) {
    p.part_max[(long long)row * p.chunks + chunk] = M;
    p.part_sum[(long long)row * p.chunks + chunk] = S;
  }
}

struct RowStats {
  float m, z, k;
};

// (max, normaliser) of a row from its chunk partials; one warp, fixed
// order, identical on every lane and in every kernel.
__device__ RowStats row_stats(const StochasticParams& p, int row, float k) {
  const int lane = threadIdx.x & 31;
  const float* pm = p.part_max + (long long)row * p.chunks;
  const float* ps = p.part_sum + (long long)row * p.chunks;
  float m = -INFINITY;
  for (int c = lane; c < p.chunks; c += 32) m = fmaxf(m, pm[c]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float z = 0.f;
  for (int c = lane; c < p.chunks; c += 32) {
    const float sc = ps[c];
    if (sc > 0.f)
      z = __fadd_rn(z, __fmul_rn(sc, exp2f(__fmul_rn(__fsub_rn(pm[c], m), k))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z = __fadd_rn(z, __shfl_xor_sync(0xffffffffu, z, o));
  return {m, z, k};
}

__device__ __forceinline__ float prob(const RowStats& r, float x) {
  return __fdiv_rn(exp2f(__fmul_rn(__fsub_rn(x, r.m), r.k)), r.z);
}

struct Walk {
  int qb, a, rejected, drej;
  RowStats fin;   // statistics of the row the next token is drawn from
};

// The accept tests, run by one full warp (every lane gets the result).
__device__ Walk walk(const StochasticParams& p, int b) {
  Walk w;
  w.qb = rows_of(p, b);
  w.a = 0;
  w.rejected = 0;
  w.drej = -1;
  if (w.qb == 0 || !(p.temperature[b] > 0.f)) {
    w.qb = 0;
    return w;
  }
  const float k = k_of(p, b);
  const int32_t* dr = p.draft_ids + (long long)b * p.q_len;
  const long long row0 = (long long)b * p.q_len;
  for (int j = 1; j < w.qb; ++j) {
    const RowStats r = row_stats(p, (int)(row0 + j - 1), k);
    const int d = dr[j];
    float pd = 0.f, qd = 1.f;
    if (d >= 0 && d < p.vocab) {
      pd = prob(r, p.logits[(row0 + j - 1) * p.vocab + d]);
      if (p.draft_probs)
        qd = p.draft_probs[((long long)b * (p.q_len - 1) + j - 1) * p.vocab + d];
    }
    const float u = p.u_accept[(long long)b * (p.q_len - 1) + j - 1];
    if (__fmul_rn(u, qd) < pd) {
      ++w.a;
    } else {
      w.rejected = 1;
      w.drej = d;
      break;
    }
  }
  w.fin = row_stats(p, (int)(row0 + w.a), k);
  return w;
}

// Draw weight of token v of the final row: p, or max(0, p - q) after a
// rejection (q one-hot at the rejected draft for a greedy drafter).
__device__ __forceinline__ float weight(const StochasticParams& p, int b,
                                        const Walk& w, bool residual,
                                        float x, int v) {
  const float pv = prob(w.fin, x);
  if (!residual) return pv;
  const float qv = p.draft_probs
      ? p.draft_probs[((long long)b * (p.q_len - 1) + w.a) * p.vocab + v]
      : (v == w.drej ? 1.f : 0.f);
  return pv > qv ? __fsub_rn(pv, qv) : 0.f;
}

__global__ void __launch_bounds__(kSampleThreads)
    residual_chunk_kernel(const StochasticParams p) {
  __shared__ float red[kSampleThreads / 32];
  __shared__ Walk s_walk;
  const int chunk = blockIdx.x, b = blockIdx.y;
  if (threadIdx.x < 32) {
    const Walk w = walk(p, b);
    if (threadIdx.x == 0) s_walk = w;
  }
  __syncthreads();
  const Walk w = s_walk;
  if (w.qb == 0 || !w.rejected) return;  // only a rejection needs W_c
  const float* x = p.logits + ((long long)b * p.q_len + w.a) * p.vocab;
  const int begin = chunk * kSampleChunk;
  const int end = min(begin + kSampleChunk, p.vocab);
  float s = 0.f;
  for (int v = begin + threadIdx.x; v < end; v += kSampleThreads)
    s = __fadd_rn(s, weight(p, b, w, true, x[v], v));
  const float W = block_sum(s, red);
  if (threadIdx.x == 0) p.chunk_w[(long long)b * p.chunks + chunk] = W;
}

__global__ void __launch_bounds__(kSampleThreads)
    sample_finalize_kernel(const StochasticParams p) {
  constexpr int kPer = kSampleChunk / kSampleThreads;  // 32 per thread
  __shared__ float red[kSampleThreads / 32];
  __shared__ float s_scan[kSampleThreads];
  __shared__ Walk s_walk;
  __shared__ int s_chunk, s_pick, s_residual;
  __shared__ float s_base, s_target;
  const int b = blockIdx.x;
  if (threadIdx.x < 32) {
    const Walk w = walk(p, b);
    if (threadIdx.x == 0) s_walk = w;
  }
  __syncthreads();
  const Walk w = s_walk;
  if (w.qb == 0) {
    if (threadIdx.x == 0) {
      p.accept_len[b] = 0;
      p.next_token[b] = -1;
      if (p.out_tokens)
        for (int j = 0; j < p.q_len; ++j)
          p.out_tokens[(long long)b * p.q_len + j] = -1;
      if (p.new_seq_lens) p.new_seq_lens[b] = p.seq_lens[b];
    }
    return;
  }
  const long long frow = (long long)b * p.q_len + w.a;
  if (threadIdx.x == 0) {
    // chunk weights: the residual's, else p's (from the row statistics);
    // a residual that sums to zero (p == q) falls back to p
    float W = 0.f;
    if (w.rejected)
      for (int c = 0; c < p.chunks; ++c)
        W = __fadd_rn(W, p.chunk_w[(long long)b * p.chunks + c]);
    const int residual = w.rejected && W > 0.f;
    const float* pm = p.part_max + frow * p.chunks;
    const float* ps = p.part_sum + frow * p.chunks;
    auto cw = [&](int c) {
      if (residual) return p.chunk_w[(long long)b * p.chunks + c];
      const float sc = ps[c];
      return sc > 0.f ? __fdiv_rn(__fmul_rn(sc, exp2f(__fmul_rn(
                                     __fsub_rn(pm[c], w.fin.m), w.fin.k))),
                                  w.fin.z)
                      : 0.f;
    };
    if (!residual) {
      W = 0.f;
      for (int c = 0; c < p.chunks; ++c) W = __fadd_rn(W, cw(c));
    }
    const float target = __fmul_rn(p.u_sample[b], W);
    float run = 0.f;
    int cs = -1;
    for (int c = 0; c < p.chunks; ++c) {
      const float nx = __fadd_rn(run, cw(c));
      if (nx > target) {
        cs = c;
        break;
      }
      run = nx;
    }
    if (cs < 0) {  // rounding put u * W at the very end: last nonzero chunk
      for (int c = p.chunks - 1; c >= 0; --c)
        if (cw(c) > 0.f) {
          cs = c;
          break;
        }
      run = -INFINITY;  // any index of that chunk qualifies; take the last
    }
    s_chunk = cs;
    s_base = run;
    s_target = target;
    s_residual = residual;
    s_pick = INT_MAX;
  }
  __syncthreads();
  const int cs = s_chunk;
  const bool residual = s_residual;
  const float* x = p.logits + frow * p.vocab;
  const int begin = cs * kSampleChunk;
  // thread t scans the kPer consecutive tokens begin + t*kPer ...
  const int v0 = begin + threadIdx.x * kPer;
  float wv[kPer];
  float tot = 0.f;
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const int v = v0 + e;
    wv[e] = v < p.vocab ? weight(p, b, w, residual, x[v], v) : 0.f;
    tot = __fadd_rn(tot, wv[e]);
  }
  // exclusive scan of the thread totals (sequential over warps, fixed order)
  s_scan[threadIdx.x] = tot;
  __syncthreads();
  if (threadIdx.x == 0) {
    float run = 0.f;
    for (int t = 0; t < kSampleThreads; ++t) {
      const float c = s_scan[t];
      s_scan[t] = run;
      run = __fadd_rn(run, c);
    }
  }
  __syncthreads();
  int found = INT_MAX, last_nz = -1;
  if (s_base == -INFINITY) {  // fallback: the chunk's last nonzero weight
#pragma unroll
    for (int e = 0; e < kPer; ++e)
      if (wv[e] > 0.f) last_nz = v0 + e;
  } else {
    float run = __fadd_rn(s_base, s_scan[threadIdx.x]);
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      run = __fadd_rn(run, wv[e]);
      if (found == INT_MAX && wv[e] > 0.f && run > s_target) found = v0 + e;
      if (wv[e] > 0.f) last_nz = v0 + e;
    }
  }
  found = __reduce_min_sync(0xffffffffu, found);
  last_nz = __reduce_max_sync(0xffffffffu, last_nz);
  if ((threadIdx.x & 31) == 0) {
    atomicMin(&s_pick, found);
    reinterpret_cast<int*>(red)[threadIdx.x >> 5] = last_nz;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int pick = s_pick;
    if (pick == INT_MAX) {  // rounding between the two sums: last nonzero
      for (int i = 0; i < kSampleThreads / 32; ++i)
        pick = pick == INT_MAX ? reinterpret_cast<int*>(red)[i]
                               : max(pick, reinterpret_cast<int*>(red)[i]);
      if (pick < 0) pick = begin;
    }
    const int32_t* dr = p.draft_ids + (long long)b * p.q_len;
    p.accept_len[b] = w.a;
    p.next_token[b] = pick;
    if (p.out_tokens) {
      int32_t* o = p.out_tokens + (long long)b * p.q_len;
      for (int j = 0; j < p.q_len; ++j)
        o[j] = j < w.a ? dr[j + 1] : (j == w.a ? pick : -1);
    }
    if (p.new_seq_lens) p.new_seq_lens[b] = p.seq_lens[b] - w.qb + w.a + 1;
  }
}

}  // namespace

cudaError_t launch_stochastic_accept(const StochasticParams& p,
                                     cudaStream_t s) {
  const int rows = p.batch * p.q_len;
  softmax_partial_kernel<<<dim3(p.chunks, rows), kSampleThreads, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  residual_chunk_kernel<<<dim3(p.chunks, p.batch), kSampleThreads, 0, s>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  sample_finalize_kernel<<<p.batch, kSampleThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace specv
