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
//   2. residual_chunk_kernel, CTA (chunk, request), only with draft
//      distributions: the accept tests (one warp per block row, all rows
//      side by side; repeated by every CTA of the request), then the
//      chunk's total draw weight max(0, p - q).  A greedy drafter (q
//      one-hot at its draft) needs no second pass: the residual is p
//      without the rejected token, whose chunk weights follow from the
//      softmax statistics;
//   3. sample_finalize_kernel, one CTA per request: the tests again, the
//      chunk that holds u * W, and a block scan of that chunk alone.
// The second and third launches are programmatic dependents of the one
// before them (scheduled while it runs, waiting for it in the kernel).
// Every float step that decides an integer goes through the same device
// functions in kernels 2 and 3 with explicitly rounded operations, so both
// see bit-identical weights.
#include <climits>

#include "common.cuh"
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
  // the residual kernel may be scheduled now; it waits for this grid
  tc_grid_launch_dependents();
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
  float m, z, k, inv_z;   // inv_z = 1/z rounded once: p(v) = e(v) * inv_z
};

// (max, normaliser) of a row from its chunk partials; one warp, fixed
// order, identical on every lane and in every kernel.  Lane l holds chunks
// l, l + 32, ... (at most kMaxSampleChunks / 32 of them): row_partials
// issues their loads, row_stats reduces them.
constexpr int kStatsPerLane = kMaxSampleChunks / 32;

__device__ __forceinline__ void row_partials(const StochasticParams& p, int row,
                                             float* cm, float* cs) {
  const int lane = threadIdx.x & 31;
  const float* pm = p.part_max + (long long)row * p.chunks;
  const float* ps = p.part_sum + (long long)row * p.chunks;
#pragma unroll
  for (int i = 0; i < kStatsPerLane; ++i) {
    const int c = lane + 32 * i;
    cm[i] = c < p.chunks ? pm[c] : -INFINITY;
    cs[i] = c < p.chunks ? ps[c] : 0.f;
  }
}

__device__ __forceinline__ RowStats row_stats(const float* cm, const float* cs,
                                              float k) {
  float m = cm[0];
#pragma unroll
  for (int i = 1; i < kStatsPerLane; ++i) m = fmaxf(m, cm[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float z = 0.f;
#pragma unroll
  for (int i = 0; i < kStatsPerLane; ++i)
    if (cs[i] > 0.f)
      z = __fadd_rn(z, __fmul_rn(cs[i], exp2f(__fmul_rn(__fsub_rn(cm[i], m), k))));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z = __fadd_rn(z, __shfl_xor_sync(0xffffffffu, z, o));
  return {m, z, k, __frcp_rn(z)};
}

__device__ __forceinline__ float prob(const RowStats& r, float x) {
  return __fmul_rn(exp2f(__fmul_rn(__fsub_rn(x, r.m), r.k)), r.inv_z);
}

struct Walk {
  int qb, a, rejected, drej;
  RowStats fin;   // statistics of the row the next token is drawn from
};

struct WalkSmem {
  RowStats stats[16];
  int ok[16];
  int d[16];      // the request's block ids: d[j + 1] is scored by row j
  float xd[16];   // row j's logit of d[j + 1] (when row j tests a draft)
  Walk walk;
};

// The accept tests of request b, run by the whole CTA: warp w takes rows
// w, w + warps, ... (their statistics and the test of the draft each row
// scores), then thread 0 counts the leading accepted drafts.  Every test is
// independent of the others, so they run side by side; the result is the
// same in every kernel that calls this.  Each row's loads that do not
// depend on its draft (the uniform, the chunk partials) are issued with the
// draft id, so a test costs two rounds of loads.  With `part` (a
// [16][kMaxSampleChunks] array) the rows' chunk partials are kept there for
// the draw.  Ends with the CTA synchronised and the walk in sm->walk.
__device__ void decide(const StochasticParams& p, int b, WalkSmem* sm,
                       float2* part) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  const long long row0 = (long long)b * p.q_len;
  const int32_t* dr = p.draft_ids + row0;
  if (threadIdx.x < p.q_len) sm->d[threadIdx.x] = dr[threadIdx.x];
  const bool live = p.temperature[b] > 0.f;
  const int qb = live ? rows_of(p, b) : 0;
  if (qb > 0) {
    const float k = k_of(p, b);
    for (int j = warp; j < qb; j += nw) {
      const bool test = j + 1 < qb;
      const int d = test ? dr[j + 1] : -1;
      const float u = test ? p.u_accept[(long long)b * (p.q_len - 1) + j] : 0.f;
      float cm[kStatsPerLane], cs[kStatsPerLane];
      row_partials(p, (int)(row0 + j), cm, cs);
      float x = 0.f, qd = 1.f;
      const bool in = test && d >= 0 && d < p.vocab;
      if (in) {
        x = p.logits[(row0 + j) * p.vocab + d];
        if (p.draft_probs)
          qd = p.draft_probs[((long long)b * (p.q_len - 1) + j) * p.vocab + d];
      }
      const RowStats r = row_stats(cm, cs, k);
      int ok = 1;
      if (test) {
        const float pd = in ? prob(r, x) : 0.f;
        ok = __fmul_rn(u, qd) < pd;   // accept draft j + 1
      }
      if (part) {
#pragma unroll
        for (int i = 0; i < kStatsPerLane; ++i)
          part[j * kMaxSampleChunks + lane + 32 * i] = make_float2(cm[i], cs[i]);
      }
      if (lane == 0) {
        sm->stats[j] = r;
        sm->ok[j] = ok;
        sm->xd[j] = x;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    Walk w;
    w.qb = qb;
    w.a = 0;
    w.rejected = 0;
    w.drej = -1;
    if (qb > 0) {
      while (w.a + 1 < qb && sm->ok[w.a]) ++w.a;
      w.rejected = w.a + 1 < qb;
      if (w.rejected) w.drej = sm->d[w.a + 1];
      w.fin = sm->stats[w.a];
    }
    sm->walk = w;
  }
  __syncthreads();
}

// Sum of the kMaxSampleChunks chunk weights in s_cw, by one warp in a fixed
// order (lane l adds chunks 4l..4l+3, then a butterfly): the same on every
// lane.
__device__ __forceinline__ float chunk_total(const float* s_cw, int lane) {
  constexpr int kPerLane = kMaxSampleChunks / 32;
  float part = 0.f;
#pragma unroll
  for (int i = 0; i < kPerLane; ++i) part = __fadd_rn(part, s_cw[lane * kPerLane + i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    part = __fadd_rn(part, __shfl_xor_sync(0xffffffffu, part, o));
  return part;
}

// Draw weight of a token of the final row, written out where it is used:
// p, or max(0, p - q) after a rejection (q one-hot at the rejected draft for
// a greedy drafter).  Both kernels evaluate the same expression.

__global__ void __launch_bounds__(kSampleThreads)
    residual_chunk_kernel(const StochasticParams p) {
  __shared__ float red[kSampleThreads / 32];
  __shared__ WalkSmem sm;
  const int chunk = blockIdx.x, b = blockIdx.y;
  tc_grid_launch_dependents();  // the draw kernel may be scheduled now
  // a programmatic dependent of the softmax pass: its partials are read
  // only once that grid is complete
  tc_grid_dependency_wait();
  decide(p, b, &sm, nullptr);
  const Walk w = sm.walk;
  if (w.qb == 0 || !w.rejected) return;  // only a rejection needs W_c
  constexpr int kPer = kSampleChunk / kSampleThreads;
  const long long frow = (long long)b * p.q_len + w.a;
  const float* x = p.logits + frow * p.vocab;
  const float* qrow = p.draft_probs
      ? p.draft_probs + ((long long)b * (p.q_len - 1) + w.a) * p.vocab
      : nullptr;
  const int begin = chunk * kSampleChunk;
  // every load of the chunk is issued before any is used
  float xv[kPer], qv[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const int v = begin + threadIdx.x + e * kSampleThreads;
    xv[e] = v < p.vocab ? x[v] : -INFINITY;
    qv[e] = qrow ? (v < p.vocab ? qrow[v] : 0.f)
                 : (v == w.drej ? 1.f : 0.f);
  }
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const float pv = prob(w.fin, xv[e]);
    s = __fadd_rn(s, pv > qv[e] ? __fsub_rn(pv, qv[e]) : 0.f);
  }
  const float W = block_sum(s, red);
  if (threadIdx.x == 0) p.chunk_w[(long long)b * p.chunks + chunk] = W;
}

__global__ void __launch_bounds__(kSampleThreads)
    sample_finalize_kernel(const StochasticParams p) {
  constexpr int kPer = kSampleChunk / kSampleThreads;  // 32 per thread
  constexpr int kWarps = kSampleThreads / 32;
  __shared__ WalkSmem sm;
  __shared__ float s_cw[kMaxSampleChunks];
  // the rows' chunk partials until the chunk weights are taken, then the
  // chosen chunk's draw weights
  __shared__ union {
    float2 part[16 * kMaxSampleChunks];
    float w[kSampleThreads * (kPer + 1)];
  } s_u;
  float* s_w = s_u.w;
  __shared__ float s_warp[kWarps];
  __shared__ int s_found[kWarps], s_last[kWarps];
  __shared__ int s_chunk, s_residual;
  __shared__ float s_base, s_target;
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // a programmatic dependent of the residual kernel (itself one of the
  // softmax pass), or of the softmax pass for a greedy drafter: everything
  // they wrote is read after this
  tc_grid_dependency_wait();
  decide(p, b, &sm, s_u.part);
  const Walk w = sm.walk;
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
  // chunk weights in shared memory: with draft distributions, the
  // residual's (from kernel 2); otherwise p's from the row statistics, and
  // after a rejection by a greedy drafter (q one-hot at the rejected draft)
  // the residual max(0, p - q) is p without the rejected token, so its
  // chunk loses that token's probability.  A zero residual (p == q) falls
  // back to p.
  const float2* fpart = s_u.part + w.a * kMaxSampleChunks;  // (max, sum)
  const bool from_kernel2 = w.rejected && p.draft_probs;
  for (int c = threadIdx.x; c < kMaxSampleChunks; c += kSampleThreads)
    s_cw[c] = from_kernel2 && c < p.chunks
                  ? p.chunk_w[(long long)b * p.chunks + c] : 0.f;
  __syncthreads();
  if (warp == 0) {
    float W = 0.f;
    bool residual = false;
    if (from_kernel2) {
      W = chunk_total(s_cw, lane);
      residual = W > 0.f;
    }
    if (!residual) {
      // the rejected draft's probability, for a greedy drafter's residual
      const bool greedy_rej = w.rejected && !p.draft_probs && w.drej >= 0 &&
                              w.drej < p.vocab;
      // (the rejecting row scored it: its logit is that row's test input)
      const float pd = greedy_rej ? prob(w.fin, sm.xd[w.a]) : 0.f;
      const int cd = greedy_rej ? w.drej / kSampleChunk : -1;
      for (int c = lane; c < kMaxSampleChunks; c += 32) {
        float v = 0.f;
        const float2 mc = fpart[c];
        if (c < p.chunks && mc.y > 0.f)
          v = __fmul_rn(__fmul_rn(mc.y, exp2f(__fmul_rn(__fsub_rn(mc.x, w.fin.m),
                                                         w.fin.k))),
                        w.fin.inv_z);
        if (c == cd) v = v > pd ? __fsub_rn(v, pd) : 0.f;
        s_cw[c] = v;
      }
      __syncwarp();
      W = chunk_total(s_cw, lane);
      if (greedy_rej) {
        residual = W > 0.f;
        if (!residual) {  // p is one-hot at the rejected draft: fall back to p
          for (int c = lane; c < kMaxSampleChunks; c += 32)
            if (c == cd) s_cw[c] = pd;
          __syncwarp();
          W = chunk_total(s_cw, lane);
        }
      }
    }
    // the first chunk whose running sum exceeds u * W: lane l scans chunks
    // 4l .. 4l+3 after an exclusive warp scan of the lanes' sums
    const float target = __fmul_rn(p.u_sample[b], W);
    constexpr int kPerLane = kMaxSampleChunks / 32;
    float cw[kPerLane], part = 0.f;
#pragma unroll
    for (int i2 = 0; i2 < kPerLane; ++i2) {
      cw[i2] = s_cw[lane * kPerLane + i2];
      part = __fadd_rn(part, cw[i2]);
    }
    float inc = part;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc = __fadd_rn(inc, y);
    }
    float run = __fsub_rn(inc, part), base = 0.f;
    int cs = INT_MAX;
#pragma unroll
    for (int i2 = 0; i2 < kPerLane; ++i2) {
      const float nx = __fadd_rn(run, cw[i2]);
      if (cs == INT_MAX && cw[i2] > 0.f && nx > target) {
        cs = lane * kPerLane + i2;
        base = run;
      }
      run = nx;
    }
    const int first = __reduce_min_sync(0xffffffffu, cs);
    int last = -1;
#pragma unroll
    for (int i2 = 0; i2 < kPerLane; ++i2)
      if (cw[i2] > 0.f) last = lane * kPerLane + i2;
    last = __reduce_max_sync(0xffffffffu, last);
    if (lane == 0) {
      s_residual = residual;
      s_target = target;
      if (first != INT_MAX) {
        s_chunk = first;
      } else {  // rounding put u * W at the very end: last nonzero chunk
        s_chunk = last >= 0 ? last : 0;
        s_base = -INFINITY;  // any index of that chunk qualifies: the last
      }
    }
    if (first != INT_MAX && cs == first) s_base = base;
  }
  __syncthreads();  // the partials are read: s_u holds the weights now
  const int cs = s_chunk;
  const bool residual = s_residual;
  const float* x = p.logits + frow * p.vocab;
  const float* qrow = residual && p.draft_probs
      ? p.draft_probs + ((long long)b * (p.q_len - 1) + w.a) * p.vocab
      : nullptr;
  const int begin = cs * kSampleChunk;
  // stage the chunk's weights in shared memory with coalesced loads, then
  // let thread t scan tokens begin + t*kPer ... (rows padded by one float
  // so the column reads hit 32 different banks)
  {
    float xv[kPer], qv[kPer];  // every load issued before any is used
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int v = begin + e * kSampleThreads + threadIdx.x;
      xv[e] = v < p.vocab ? x[v] : -INFINITY;
      qv[e] = qrow ? (v < p.vocab ? qrow[v] : 0.f)
                   : (residual && v == w.drej ? 1.f : 0.f);
    }
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int i2 = e * kSampleThreads + threadIdx.x;
      const float pv = prob(w.fin, xv[e]);
      s_w[(i2 / kPer) * (kPer + 1) + i2 % kPer] =
          !residual ? pv : (pv > qv[e] ? __fsub_rn(pv, qv[e]) : 0.f);
    }
  }
  __syncthreads();
  const int v0 = begin + threadIdx.x * kPer;
  const float* mine = s_w + threadIdx.x * (kPer + 1);
  float tot = 0.f;
#pragma unroll
  for (int e = 0; e < kPer; ++e) tot = __fadd_rn(tot, mine[e]);
  // exclusive prefix of the thread totals: warp shuffle scan, then the warp
  // totals in order (a fixed pattern, so the same sums every time)
  float inc = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc = __fadd_rn(inc, y);
  }
  if (lane == 31) s_warp[warp] = inc;
  __syncthreads();
  float wbase = 0.f;
  for (int i2 = 0; i2 < warp; ++i2) wbase = __fadd_rn(wbase, s_warp[i2]);
  const float excl = __fadd_rn(wbase, __fsub_rn(inc, tot));
  int found = INT_MAX, last_nz = -1;
  if (s_base == -INFINITY) {  // fallback: the chunk's last nonzero weight
#pragma unroll
    for (int e = 0; e < kPer; ++e)
      if (mine[e] > 0.f) last_nz = v0 + e;
  } else {
    float run = __fadd_rn(s_base, excl);
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      run = __fadd_rn(run, mine[e]);
      if (found == INT_MAX && mine[e] > 0.f && run > s_target) found = v0 + e;
      if (mine[e] > 0.f) last_nz = v0 + e;
    }
  }
  found = __reduce_min_sync(0xffffffffu, found);
  last_nz = __reduce_max_sync(0xffffffffu, last_nz);
  if (lane == 0) {
    s_found[warp] = found;
    s_last[warp] = last_nz;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int pick = INT_MAX, last = -1;
    for (int i2 = 0; i2 < kWarps; ++i2) {
      pick = min(pick, s_found[i2]);
      last = max(last, s_last[i2]);
    }
    if (pick == INT_MAX)  // rounding between the two sums: last nonzero
      pick = last >= 0 ? last : begin;
    p.accept_len[b] = w.a;
    p.next_token[b] = pick;
    if (p.out_tokens) {
      int32_t* o = p.out_tokens + (long long)b * p.q_len;
      for (int j = 0; j < p.q_len; ++j)
        o[j] = j < w.a ? sm.d[j + 1] : (j == w.a ? pick : -1);
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
  // the second and third launches are programmatic dependents of the one
  // before: they are scheduled while it runs and wait for it in the kernel
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kSampleThreads);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.draft_probs) {  // a greedy drafter's residual needs no second pass
    cfg.gridDim = dim3(p.chunks, p.batch);
    e = cudaLaunchKernelEx(&cfg, residual_chunk_kernel, p);
    if (e != cudaSuccess) return e;
  }
  cfg.gridDim = dim3(p.batch);
  return cudaLaunchKernelEx(&cfg, sample_finalize_kernel, p);
}

}  // namespace specv
