// DFlash2 candidate selection ("MTP and DFlash2 at long context on XPU",
// "The part that makes DFlash2 different" and "Selector and recurrent math";
// "Qwen3.8-27B-FP8" page: selector_rank 256, selector_top_k 16, an exact
// MAP over the chain as an option).
//
// Draft position t = 1 .. P-1 keeps its K best candidate logits (larger
// first, lower token id on ties).  A transition from candidate a at t-1 (the
// boundary token at t = 1) to candidate b at t scores
//     S_t(a, b) = U_t(b) + sum_r A[a, r] H_t[r] B[b, r],   H_t = W_H h_t,
// and a walk from the boundary picks one chain: greedy (the best successor
// of the token already chosen) or MAP (the best total score).  Ties go to
// the lower candidate rank.
//
// Three launches (after a reset of the per-request counters):
//   1. topk_partial_kernel, CTA per (8192-token chunk, position row): the
//      chunk's K best in one streaming pass (K rounds of warp argmax over
//      register-held logits, then a block merge);
//   2. project_kernel: H = W_H h for every position row, bf16 mma.sync
//      tiles with fp32 accumulation (a small contraction: the weights are
//      read once);
//   3. table_kernel, CTA per (position, request): the candidate lists of t
//      and t-1 from the chunk lists, the 2 x K codebook rows, and the K x K
//      table in fp32; the request's last CTA to finish (a counter) then
//      walks the chain, greedy or MAP, with one warp.
#include <climits>

#include "common.cuh"
#include "selector.cuh"

namespace specv {
namespace {

// Larger value first, then lower token id: a total order on distinct ids.
__device__ __forceinline__ bool better(float a, int ia, float b, int ib) {
  return a > b || (a == b && ia < ib);
}

__device__ __forceinline__ void warp_best(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (better(ov, oi, v, i)) {
      v = ov;
      i = oi;
    }
  }
}

// ---- 1. chunk top-K -------------------------------------------------------

// Exact top-K of a chunk (K <= 16) without serial rounds.  (i) A bound:
// each of the 8 warps holds two values at or above its second largest lane
// maximum, so the chunk holds 16 >= K values at or above the smallest of
// those, T, and its K best all lie at or above T.  (ii) The values >= T
// (under 1% of a chunk of random logits) go to a shared pool, and each pool
// entry's rank is the number of entries that beat it (value, then lower
// token id): entries of rank < K are the chunk's top K, already in order.  A pool that overflows (heavy ties, or fewer than K finite values)
// falls back to K block-wide argmax rounds over the whole chunk.
constexpr int kSelPool = 512;

// Four CTAs per SM (64 registers, a few bytes of spill): the pass waits on
// memory, and the extra resident CTA keeps more loads in flight than the
// spill costs (three CTAs at 80 registers, or five at 48 with more spill,
// measured slower).
__global__ void __launch_bounds__(kSelThreads, 4)
    topk_partial_kernel(const SelectParams p) {
  constexpr int kPer = kSelChunk / kSelThreads;  // 32 logits per thread
  constexpr int kWarps = kSelThreads / 32;
  __shared__ float s_tw[kWarps];
  __shared__ float s_pv[kSelPool];
  __shared__ int s_pi[kSelPool];
  __shared__ int s_n;
  // the projection kernel may start now: it reads none of this kernel's
  // output and runs alongside it
  tc_grid_launch_dependents();
  const int chunk = blockIdx.x, row = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* x = p.cand_logits + (long long)row * p.vocab;
  const int begin = chunk * kSelChunk;
  const int end = min(begin + kSelChunk, p.vocab);
  // thread t holds tokens begin + 4 (t + 256 e) + q, q < 4, e < 8
  float v[kPer];
  if (p.vec4) {
    const float4* x4 = reinterpret_cast<const float4*>(x + begin);
    const int n4 = (end - begin) >> 2;
#pragma unroll
    for (int e = 0; e < kPer / 4; ++e) {
      const int j = threadIdx.x + e * kSelThreads;
      const float4 t = j < n4 ? __ldcs(x4 + j)
                              : make_float4(-INFINITY, -INFINITY, -INFINITY,
                                            -INFINITY);
      v[4 * e] = t.x; v[4 * e + 1] = t.y; v[4 * e + 2] = t.z; v[4 * e + 3] = t.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < kPer / 4; ++e) {
      const int i0 = begin + 4 * (threadIdx.x + e * kSelThreads);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        v[4 * e + q] = i0 + q < end ? __ldcs(x + i0 + q) : -INFINITY;
    }
  }
  auto id_of = [&](int e) {
    const int id = begin + 4 * (threadIdx.x + (e >> 2) * kSelThreads) + (e & 3);
    return id < end ? id : INT_MAX;
  };
  // (i) the bound: every warp holds two values at or above its second
  // largest lane maximum, so the 8 warps hold 16 >= K values at or above
  // the smallest of those
  float m = v[0];
#pragma unroll
  for (int e = 1; e < kPer; ++e) m = fmaxf(m, v[e]);
  float m1 = m;
  int l1 = lane;
  warp_best(m1, l1);
  float m2 = lane == l1 ? -INFINITY : m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m2 = fmaxf(m2, __shfl_xor_sync(0xffffffffu, m2, o));
  if (lane == 0) s_tw[warp] = m2;
  if (threadIdx.x == 0) s_n = 0;
  __syncthreads();
  float T = s_tw[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) T = fminf(T, s_tw[w]);
  // (ii) the pool of values >= T
  const bool finite_bound = T > -INFINITY;
  if (finite_bound) {
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      if (v[e] >= T) {
        const int slot = atomicAdd(&s_n, 1);
        if (slot < kSelPool) {
          s_pv[slot] = v[e];
          s_pi[slot] = id_of(e);
        }
      }
    }
  }
  __syncthreads();
  const int n = s_n;
  float* ov = p.part_val + ((long long)row * p.chunks + chunk) * p.top;
  int32_t* oi = p.part_idx + ((long long)row * p.chunks + chunk) * p.top;
  if (finite_bound && n <= kSelPool) {
    for (int e = threadIdx.x; e < n; e += kSelThreads) {
      const float ve = s_pv[e];
      const int ie = s_pi[e];
      int r = 0;
      for (int f = 0; f < n; ++f) r += better(s_pv[f], s_pi[f], ve, ie);
      if (r < p.top) {
        ov[r] = ve;
        oi[r] = ie;
      }
    }
    return;
  }
  // fallback: K block-wide argmax rounds over every value of the chunk
  __shared__ float s_bv[kWarps];
  __shared__ int s_bi[kWarps];
  uint32_t taken = 0;
  for (int k = 0; k < p.top; ++k) {
    float bv = -INFINITY;
    int bi = INT_MAX;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int id = id_of(e);
      if (!(taken >> e & 1u) && id != INT_MAX && better(v[e], id, bv, bi)) {
        bv = v[e];
        bi = id;
      }
    }
    warp_best(bv, bi);
    if (lane == 0) {
      s_bv[warp] = bv;
      s_bi[warp] = bi;
    }
    __syncthreads();
    float wv = s_bv[0];
    int wi = s_bi[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w)
      if (better(s_bv[w], s_bi[w], wv, wi)) {
        wv = s_bv[w];
        wi = s_bi[w];
      }
    __syncthreads();
    if (threadIdx.x == 0) {
      ov[k] = wv;
      oi[k] = wi;
    }
    if (wi != INT_MAX)
#pragma unroll
      for (int e = 0; e < kPer; ++e)
        if (id_of(e) == wi) taken |= 1u << e;
  }
}

// ---- 2. projection H = W_H h ---------------------------------------------------

__device__ __forceinline__ void mma_bf16_16816(float* c, const uint32_t* a,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

constexpr int kProjMTiles = 4;  // 64 rows of h per CTA

// CTA (n tile of 8 projection rows, m block of 64 position rows, k slice z
// of 128 columns); warp w takes the slice's k16 step w alone, so all of its
// fragment loads are in flight together; the 8 warps' tiles are summed in a
// fixed order into the slice's partial, and the table kernel sums the
// D / 128 slices in a fixed order.
__global__ void __launch_bounds__(256) project_kernel(const SelectParams p) {
  __shared__ float s_acc[8][kProjMTiles * 16][8];
  tc_grid_launch_dependents();  // the table kernel may be scheduled now
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int n0 = blockIdx.x * 8, m0 = blockIdx.y * kProjMTiles * 16;
  const int rows = p.batch * (p.positions - 1);
  const uint32_t* W = reinterpret_cast<const uint32_t*>(p.w_h);
  const uint32_t* X = reinterpret_cast<const uint32_t*>(p.hidden);
  const int d2 = p.dim >> 1;  // bf16 pairs per row
  float acc[kProjMTiles][4];
#pragma unroll
  for (int m = 0; m < kProjMTiles; ++m)
    acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.f;
  const int ksteps = p.dim >> 4;
  const int n = n0 + g;
  {
    const int ks = blockIdx.z * 8 + warp;
    const int kp = ks * 8 + t4;  // pair index of columns 16 ks + 2 t4
    uint32_t b0 = 0, b1 = 0;
    if (n < p.rank && ks < ksteps) {
      b0 = W[(long long)n * d2 + kp];
      b1 = W[(long long)n * d2 + kp + 4];
    }
#pragma unroll
    for (int m = 0; m < kProjMTiles; ++m) {
      const int r0 = m0 + m * 16 + g, r1 = r0 + 8;
      uint32_t a[4] = {0u, 0u, 0u, 0u};
      if (r0 < rows && ks < ksteps) {
        a[0] = X[(long long)r0 * d2 + kp];
        a[2] = X[(long long)r0 * d2 + kp + 4];
      }
      if (r1 < rows && ks < ksteps) {
        a[1] = X[(long long)r1 * d2 + kp];
        a[3] = X[(long long)r1 * d2 + kp + 4];
      }
      mma_bf16_16816(acc[m], a, b0, b1);
    }
  }
#pragma unroll
  for (int m = 0; m < kProjMTiles; ++m) {
    s_acc[warp][m * 16 + g][2 * t4] = acc[m][0];
    s_acc[warp][m * 16 + g][2 * t4 + 1] = acc[m][1];
    s_acc[warp][m * 16 + g + 8][2 * t4] = acc[m][2];
    s_acc[warp][m * 16 + g + 8][2 * t4 + 1] = acc[m][3];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < kProjMTiles * 16 * 8; e += 256) {
    const int r = e >> 3, c = e & 7;
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += s_acc[w][r][c];
    if (m0 + r < rows && n0 + c < p.rank)
      p.proj[((long long)blockIdx.z * rows + m0 + r) * p.rank + n0 + c] = s;
  }
  // launched as a programmatic dependent of the top-K pass, which it does
  // not read: it waits for that grid only here, so that this grid completes
  // after it and the table kernel (waiting for this grid) sees both
  tc_grid_dependency_wait();
}

// ---- 3. transition tables ---------------------------------------------------

// The K best of a position row from its chunk lists, by one warp (every lane
// gets the same lists); ids[k], vals[k] in smem.  Lane c holds chunk c's
// sorted list as a register queue (one round of loads); each round the
// lanes offer their heads and the winner shifts its queue.
__device__ void merge_candidates(const SelectParams& p, int row, int* ids,
                                 float* vals) {
  const int lane = threadIdx.x & 31;
  float qv[16];
  int qi[16];
  const float* pv = p.part_val + ((long long)row * p.chunks + lane) * p.top;
  const int32_t* pi = p.part_idx + ((long long)row * p.chunks + lane) * p.top;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const bool ok = lane < p.chunks && k < p.top;
    qv[k] = ok ? pv[k] : -INFINITY;
    qi[k] = ok ? pi[k] : INT_MAX;
  }
  for (int k = 0; k < p.top; ++k) {
    float wv = qv[0];
    int wi = qi[0];
    warp_best(wv, wi);
    if (lane == 0) {
      ids[k] = wi == INT_MAX ? -1 : wi;
      vals[k] = wv;
    }
    if (wi != INT_MAX && wi == qi[0]) {
#pragma unroll
      for (int e = 0; e < 15; ++e) {
        qv[e] = qv[e + 1];
        qi[e] = qi[e + 1];
      }
      qv[15] = -INFINITY;
      qi[15] = INT_MAX;
    }
  }
}

// ---- 4. the walk -------------------------------------------------------------

// Request b's tables and candidates into shared memory (s_tr >= (P-1) K K
// floats, s_ci >= (P-1) K ints), by the whole CTA.  Other CTAs wrote them
// (ordered by their fence and count): they are read from L2, every load of a
// thread issued before any is stored.  P-1 <= 15 and K <= 16, so a thread
// of the 256 holds at most 15 table entries and one candidate.
__device__ __forceinline__ void stage_walk(const SelectParams& p, int b,
                                           float* s_tr, int* s_ci) {
  const int P1 = p.positions - 1, K = p.top;
  const int ntr = P1 * K * K, nci = P1 * K;
  const float* tr = p.trans + (long long)b * ntr;
  const int32_t* ci = p.cand_ids + (long long)b * nci;
  float v[15];
#pragma unroll
  for (int i = 0; i < 15; ++i) {
    const int e = threadIdx.x + 256 * i;
    v[i] = e < ntr ? __ldcg(tr + e) : 0.f;
  }
  const int c = (int)threadIdx.x < nci ? __ldcg(ci + threadIdx.x) : 0;
#pragma unroll
  for (int i = 0; i < 15; ++i) {
    const int e = threadIdx.x + 256 * i;
    if (e < ntr) s_tr[e] = v[i];
  }
  if ((int)threadIdx.x < nci) s_ci[threadIdx.x] = c;
}

// The greedy or MAP walk of request b by one warp, from the tables and
// candidates staged in shared memory (s_back >= 16 x 16 ints).
__device__ void walk_request(const SelectParams& p, int b, const float* s_tr,
                             const int* s_ci, int* s_back) {
  const int lane = threadIdx.x & 31;
  const int P1 = p.positions - 1, K = p.top;
  int32_t* out = p.draft_ids + (long long)b * p.positions;
  if (lane == 0) out[0] = p.boundary[b];
  if (p.mode == 0) {  // greedy
    int prev = 0;
    for (int t = 1; t <= P1; ++t) {
      float v = lane < K ? s_tr[((t - 1) * K + prev) * K + lane] : -INFINITY;
      int i = lane < K ? lane : INT_MAX;
      warp_best(v, i);
      prev = i;
      if (lane == 0) out[t] = s_ci[(t - 1) * K + prev];
    }
    return;
  }
  // MAP: best_t(c) = max_a best_{t-1}(a) + S_t(a, c), lowest a on ties
  float best = lane < K ? s_tr[lane] : -INFINITY;  // t = 1 from the boundary
  for (int t = 2; t <= P1; ++t) {
    float nb = -INFINITY;
    int arg = 0;
    for (int a2 = 0; a2 < K; ++a2) {
      const float ba = __shfl_sync(0xffffffffu, best, a2);
      const float w = lane < K
          ? __fadd_rn(ba, s_tr[((t - 1) * K + a2) * K + lane])
          : -INFINITY;
      if (a2 == 0 || w > nb) {
        nb = w;
        arg = a2;
      }
    }
    if (lane < K) s_back[(t - 1) * 16 + lane] = arg;
    best = nb;
  }
  float v = best;
  int c = lane < K ? lane : INT_MAX;
  warp_best(v, c);
  __syncwarp();
  if (lane == 0) {
    for (int t = P1; t >= 1; --t) {
      out[t] = s_ci[(t - 1) * K + c];
      if (t > 1) c = s_back[(t - 1) * 16 + c];
    }
  }
}

__global__ void __launch_bounds__(256) table_kernel(const SelectParams p) {
  __shared__ int s_ids[2][16];
  __shared__ float s_vals[2][16];
  __shared__ float s_ah[kSelMaxRank][17];  // A[a, r] H_t[r], column a
  __shared__ float s_b[kSelMaxRank][17];   // B[c, r], column c
  __shared__ float s_h[kSelMaxRank];
  const int t = blockIdx.x + 1, b = blockIdx.y;  // position t = 1 .. P-1
  const int P1 = p.positions - 1, K = p.top, R = p.rank;
  const int row = b * P1 + t - 1;
  // candidate lists of t (warp 0) and t-1 (warp 1), side by side with
  // H_t = the sum of the projection's k slices in slice order (warps 2..7)
  const int warp = threadIdx.x >> 5;
  const int rows = p.batch * P1;
  // a programmatic dependent of the projection kernel, whose completion
  // follows the top-K pass's: both grids' outputs are read after this
  tc_grid_dependency_wait();
  if (warp == 0) {
    merge_candidates(p, row, s_ids[1], s_vals[1]);
  } else if (warp == 1) {
    if (t > 1) merge_candidates(p, row - 1, s_ids[0], s_vals[0]);
    else if (threadIdx.x == 32) s_ids[0][0] = p.boundary[b];
  } else {
    const int slices = (p.dim + 127) >> 7;
    for (int r = threadIdx.x - 64; r < R; r += 192) {
      float hv = 0.f;
#pragma unroll 20
      for (int z = 0; z < slices; ++z)
        hv += p.proj[((long long)z * rows + row) * R + r];
      s_h[r] = hv;
    }
  }
  __syncthreads();
  const int n_pred = t == 1 ? 1 : K;
  // gather the codebook rows (all loads issued first): predecessors scaled
  // by H_t, successors as they are
  constexpr int kIt = 16 * kSelMaxRank / 256;
  __nv_bfloat16 ga[kIt], gb[kIt];
#pragma unroll
  for (int it = 0; it < kIt; ++it) {
    const int e = threadIdx.x + it * 256;
    const int a = e / R, r = e - a * R;
    const bool in = e < 16 * R;
    ga[it] = in && a < n_pred && s_ids[0][a] >= 0
                 ? p.code_a[(long long)s_ids[0][a] * R + r]
                 : __float2bfloat16(0.f);
    gb[it] = in && a < K && s_ids[1][a] >= 0
                 ? p.code_b[(long long)s_ids[1][a] * R + r]
                 : __float2bfloat16(0.f);
  }
#pragma unroll
  for (int it = 0; it < kIt; ++it) {
    const int e = threadIdx.x + it * 256;
    if (e < 16 * R) {
      const int a = e / R, r = e - a * R;
      s_ah[r][a] = __fmul_rn(__bfloat162float(ga[it]), s_h[r]);
      s_b[r][a] = __bfloat162float(gb[it]);
    }
  }
  __syncthreads();
  const int a = threadIdx.x >> 4, c = threadIdx.x & 15;
  if (a < K && c < K) {
    float s = -INFINITY;
    if (a < n_pred) {
      // four interleaved partial sums (ranks r = 4i + j), added in a fixed
      // order: four independent chains of fused multiply-adds
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      int r = 0;
      for (; r + 4 <= R; r += 4) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          acc[j] = fmaf(s_ah[r + j][a], s_b[r + j][c], acc[j]);
      }
      for (; r < R; ++r) acc[0] = fmaf(s_ah[r][a], s_b[r][c], acc[0]);
      s = s_vals[1][c] + ((acc[0] + acc[1]) + (acc[2] + acc[3]));
    }
    p.trans[(((long long)b * P1 + t - 1) * K + a) * K + c] = s;
    if (a == 0) {
      p.cand_ids[((long long)b * P1 + t - 1) * K + c] = s_ids[1][c];
      p.cand_logit[((long long)b * P1 + t - 1) * K + c] = s_vals[1][c];
    }
  }
  // the request's last table CTA to finish walks the chain
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0)
    s_last = atomicAdd(&p.counters[b], 1) == P1 - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  stage_walk(p, b, &s_ah[0][0], reinterpret_cast<int*>(&s_b[0][0]));
  __syncthreads();
  if (warp == 0)
    walk_request(p, b, &s_ah[0][0], reinterpret_cast<int*>(&s_b[0][0]),
                 reinterpret_cast<int*>(&s_b[0][0]) + 15 * 16);
}

}  // namespace

cudaError_t launch_dflash2_select(const SelectParams& p, cudaStream_t s) {
  const int rows = p.batch * (p.positions - 1);
  topk_partial_kernel<<<dim3(p.chunks, rows), kSelThreads, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // the projection and the table kernel are programmatic dependents of the
  // launch before them: the projection overlaps the top-K pass, the table
  // kernel is scheduled while the projection runs
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3((p.rank + 7) / 8,
                     (rows + kProjMTiles * 16 - 1) / (kProjMTiles * 16),
                     (p.dim + 127) / 128);
  e = cudaLaunchKernelEx(&cfg, project_kernel, p);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(p.positions - 1, p.batch);
  return cudaLaunchKernelEx(&cfg, table_kernel, p);
}

}  // namespace specv
