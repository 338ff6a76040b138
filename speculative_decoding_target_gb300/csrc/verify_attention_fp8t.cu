// Split-KV paged GQA verify attention for FP8-E4M3 KV with fp16 scales
// ("Qwen3.8-27B-FP8" page, "Implemented execution path": E4M3 cache with
// per-token / per-KV-head FP16 scales over 64-channel blocks), for blocks of
// at most 64 query rows per KV head, on the tcgen05 tensor cores with both
// KV operands held in tensor memory.
//
// The attention of one (request, KV head) piece is computed transposed:
//   S^T = K Q^T      M = 128 cached tokens, N = NR query rows, K = channels
//   O^T += V^T P^T   M = 128 channels (two halves), N = NR rows, K = tokens
// so the MMA's 128-row dimension is filled with keys or channels and its
// N dimension is the verify block's own q_len x group rows ("MTP and DFlash2
// at long context on XPU", Part III: the block's query positions folded into
// the head dimension, so each KV byte is read once).  The dequantised K tile
// and the transposed V tile are written by the dequant warps straight into
// tensor memory as A operands, so the fp16 copies never pass through shared
// memory: per 128 tokens, shared memory carries the staged FP8 bytes (TMA
// write + one read), the Q and P operand reads of the MMAs and the P
// stores, about half the traffic of dequantising into shared-memory
// operands.  NR = q_len x group rounded up to 16.
//
// Tensor memory (512 columns; NR = rows rounded up to 16, at most 64):
//   [0, 128)    K tile: lane = token, column c = channels 2c (low), 2c + 1
//   [128, ...)  V^T slots of 64 tokens (three when NR <= 48, else two), 64
//               columns each: half h at + 32 h; lane = channel 128 h + lane,
//               column c = tokens 2c (low), 2c + 1
//   then O^T (half h at + h NR; lane = channel, column = row) and two S^T
//   buffers of NR columns (lane = token, column = row).
//
// Shared memory: 2-slot rings of staged K bytes (+ scales) and of staged V
// bytes (+ scales): K is converted first and its slot released early, V is
// held until its conversion ends.  Then Q (the QK^T B operand) and two P^T
// buffers (the PV B operand).
//
// Warp roles (512 threads; 128 registers each):
//   warps 0..3    softmax: one thread per token lane.  One pass per tile
//                 loads S^T_j in 16-column chunks, masks it and writes
//                 P^T_j = 2^(s - m) (fp16) to shared memory with a running
//                 maximum m per row shared by all 128 threads, noting any
//                 score that passes it by more than 2^8; after a vote of the
//                 four warps such a tile (rarely) raises m, rescales O^T and
//                 the partial sums and is written again.  Each thread then
//                 adds its fp16 P^T row to per-thread partial row sums; the
//                 epilogue sums them over the tokens, reads O^T and writes
//                 the bf16 output or an fp32 partial.
//   warps 4..11   dequant, two sets of four warps taking alternate tiles:
//                 token lane L converts K row L into TMEM lane L
//                 (fp16(e4m3 * scale)); then, per 64-token V^T slot, a
//                 transposing 16 x 16 byte-matrix load hands thread 4 g + j
//                 channel g (and g + 8) of four consecutive tokens, which
//                 after the conversion is the register layout of a 16-lane x
//                 256-bit TMEM store (lane = channel, column = token pair).
//   warp 12       producer: per 128-token tile, lane i loads page run i
//                 (min(page_size, 64) tokens): 2-D TMA boxes of 128 bytes x
//                 run with the 128-byte swizzle for each half of the K and V
//                 rows, and 1-D bulk copies of the run's scales.
//   warp 13       QK^T issuer (one thread): S^T_j, 16 MMAs, A = K tile in
//                 TMEM, B = Q from shared memory.
//   warp 14       PV issuer (one thread): O^T += V^T_j P^T_j per 64-token
//                 slot, 2 x 4 MMAs, A = V^T slot in TMEM, B = P^T.
//   The two issuers wait (bounded) for their own inputs in tile order, so a
//   ready PV never waits behind a QK^T issue.
//
// Every wait is bounded (AttnParams::wait_cycles, about two seconds by
// default); a wait that runs out sets SPEC_STATUS_TIMEOUT in the status word
// (checked mode) and makes every later wait of the CTA return at once, so
// the kernel always finishes.  The producer then issues no further loads,
// and the teardown waits (with the long bound) for the loads, bulk stores
// and MMAs already issued before it frees tensor memory.
#include <cuda_fp8.h>

#include <cstddef>

#include "common.cuh"
#include "spec_verify.h"
#include "tc_ptx.cuh"
#include "tmem_io.cuh"

namespace specv {
namespace {

constexpr int kTile = 128;                  // tokens per tile
// Staging: separate rings for the K and the V bytes of a tile, so the K
// slot, converted first, is refilled while V is still being converted.
constexpr int kHalf = kTile * 128;          // 128-channel half of K or V
constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr int kSBytes = 2 * kHalf;          // K or V bytes, two halves
constexpr int kKSlot = kSBytes + kTile * 8;             // + K scales
constexpr int kVSlot = kSBytes + kTile * 8 + kTile * 8;  // + V scales, transposed
constexpr int kOffKS = kSBytes;             // scales [token][4] fp16 in a slot
constexpr int kOffVT = kSBytes + kTile * 8; // V scales [4][token] (dequant)
constexpr int kOffKR = 0;                   // K ring
constexpr int kOffVR = kKStages * kKSlot;   // V ring
constexpr int kRowsMax = 64;                // NR of the largest instance
constexpr int kOffQ = kOffVR + kVStages * kVSlot;
constexpr int kOffP = kOffQ + kRowsMax * 512;
constexpr int kPBytes = kTile * 128;        // one of two P^T buffers
constexpr int kOffRed = kOffP + 2 * kPBytes;
constexpr uint32_t kColK = 0, kColV = 128;
constexpr int kSub = 64;                    // tokens per V^T slot
// Tensor-memory columns of the NR-row instance: V^T slots of 64 tokens
// (three when NR <= 48, so V of the next tile is converted while PV of the
// current one runs; two at NR = 64), then O^T and the S^T buffers.
template <int NR>
struct Cols {
  static constexpr int kVSlots = NR <= 48 ? 3 : 2;
  static constexpr uint32_t kO = kColV + 64 * kVSlots;  // O^T half h: kO + h NR
  static constexpr uint32_t kS = kO + 2 * NR;           // S^T buffer b: kS + b NR
  static_assert(kS + 2 * NR <= 512, "tensor memory holds 512 columns");
};
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kThreads = 512;
constexpr int kPieceThreads = 6 * 32;       // warps 0..3, 13 and 14
constexpr int kWarpProducer = 12, kWarpQK = 13, kWarpPV = 14;
static_assert(kKSlot % 1024 == 0 && kVSlot % 1024 == 0 && kOffQ % 1024 == 0 &&
                  kOffP % 1024 == 0,
              "swizzled operands need 1024-byte alignment");

// Softmax exchange area (shared memory).
struct Red {
  float colmax[4][kRowsMax];  // per-warp column maxima of raw scores
  float m[2][kRowsMax];       // running maximum (base 2), two generations
  float mu[2][kRowsMax];      // the same with -inf replaced by 0
  float alpha[kRowsMax];      // rescale factor of the last update
  float lsum_w[4][kRowsMax];  // per-warp row sums
  float lsum[kRowsMax];
  int lim[kRowsMax];          // causal limit of each row in this piece
  float inv[kRowsMax];        // 1 / row sum (0 for a row with no key)
  long long out_off[kRowsMax];  // output row offset (elements), -1: none
  int flag[2][4];
};
static_assert(offsetof(Red, inv) % 16 == 0 && offsetof(Red, out_off) % 16 == 0,
              "the epilogue reads the row constants as 16-byte vectors");
constexpr int kOffPre = kOffRed + (int)((sizeof(Red) + 127) / 128 * 128);
constexpr int kPreBytes = ((kMaxBatch + 1) * 4 + 127) / 128 * 128;
constexpr int kSmem = kOffPre + kPreBytes + 1024;  // + alignment slack

struct Bars {
  uint64_t k8_full[kKStages];  // staged K bytes landed (TMA / bulk tx)
  uint64_t k8_empty[kKStages]; // dequant warps done with the K slot
  uint64_t v8_full[kVStages];  // staged V bytes landed
  uint64_t v8_empty[kVStages]; // dequant warps done with the V slot
  // The K tile in two channel halves, so the next tile's first half is
  // written while the last eight MMAs of QK^T read the second half:
  uint64_t k_full_a;           // channels 0..127 of K written to TMEM
  uint64_t k_full;             // channels 128..255 written (the whole tile)
  // QK^T's first eight MMAs (channels 0..127) of tile j done: that half
  // may be rewritten.  One barrier per dequant set: QK^T of tile j commits
  // to the barrier of the set that writes tile j + 1, so each barrier has
  // one waiter that consumes its phases in order (a barrier shared by the
  // two sets could be waited for a phase it has not reached, which a
  // parity wait mistakes for complete).
  uint64_t k_free_a[2];
  uint64_t v_full[3];          // V^T slot written to TMEM
  // PV of the slot's 64 tokens complete, one barrier per slot and dequant
  // set: PV commits to the set that writes the slot next, so each barrier
  // has one waiter that consumes every phase in order.  (A barrier shared
  // by the two sets, which take alternate tiles, can be waited for a phase
  // two ahead of it, which a parity wait mistakes for complete.)
  uint64_t v_empty[3][2];
  uint64_t s_full[2];          // S^T_j complete (also: K tile free again)
  uint64_t p_full[2];          // P^T_j in shared memory (S^T_j consumed)
  uint64_t pv_done[2];         // O^T += V^T_j P^T_j complete
  uint64_t drain;
};

struct Ctx {
  Bars* bars;
  volatile int* abort;
  const AttnParams* p;
  void* smem;  // 1024-byte aligned dynamic shared memory
};

struct Piece {
  int b, g, nt, len, tok_begin, tok_end, n_tiles;
  long long s0;
};

// The teardown's drain (ignore_abort) keeps the long bound whatever the
// main-loop bound is: copies and MMAs already issued must land before the
// CTA frees its tensor memory and exits.  Inlined: a call would make the
// softmax warps save their live registers around every wait.
__device__ __forceinline__ bool wait_slow(uint32_t a, uint32_t parity,
                                       volatile int* abort,
                                       const AttnParams* p, bool ignore_abort) {
  if (!ignore_abort && *abort) return false;
  const long long bound = ignore_abort ? kDrainWaitCycles : p->wait_cycles;
  const long long t0 = clock64();
  while (true) {
    if (tc::bar_try_wait(a, parity)) return true;
    if (!ignore_abort && *abort) return false;
    if (clock64() - t0 > bound) {
      *abort = 1;
      if (p->status) atomicOr(p->status, SPEC_STATUS_TIMEOUT);
      return false;
    }
  }
}
__device__ __forceinline__ bool wait_bar(const Ctx& cx, uint64_t* bar,
                                         uint32_t parity,
                                         bool ignore_abort = false) {
  const uint32_t a = tc::smem_u32(bar);
  if (tc::bar_try_wait(a, parity)) return true;
  return wait_slow(a, parity, cx.abort, cx.p, ignore_abort);
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

// Bulk store of shared-memory bytes to global memory through the async
// proxy, tracked in this thread's bulk async-groups.
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src,
                                           uint32_t bytes) {
  asm volatile(
      "cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n"
      "cp.async.bulk.commit_group;" ::"l"(dst),
      "r"(src), "r"(bytes)
      : "memory");
}
// Wait until this thread's bulk stores have read their shared-memory
// source (the buffer may be rewritten) or, with kDone, have completed.
template <bool kDone>
__device__ __forceinline__ void bulk_store_wait() {
  if (kDone)
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  else
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src,
                                          uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// ---- warp 0: staging of the piece's FP8 tiles ------------------------------
__device__ __forceinline__ int box_page(const AttnParams& p, const Piece& pc,
                                        int jt, int lane) {
  const int t = pc.tok_begin + jt * kTile + lane * p.box_rows;
  if (jt >= pc.n_tiles || t >= pc.tok_end || lane * p.box_rows >= kTile)
    return 0;
  int page = __ldg(p.page_table + (long long)pc.b * p.max_pages +
                   (t >> p.log2_ps));
  if (page < 0 || page >= p.num_pages) {
    if (p.status) atomicOr(p.status, SPEC_STATUS_BAD_PAGE);
    page = 0;  // in bounds; the affected rows are unspecified
  }
  return page;
}

// Returns false once the CTA gave up (a wait ran out): from then on no load
// is issued, and *last_k / *last_v hold the last tiles whose K / V loads
// were issued, so that the teardown waits for exactly the loads in flight.
// A slot is refilled only once its previous tile's bytes have landed and
// been consumed, so at most one load per slot is ever in flight.
__device__ bool produce(const Ctx& cx, const Piece& pc, int gj0, uint8_t* smem,
                        const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                        int* last_k, int* last_v) {
  const AttnParams& p = *cx.p;
  const int lane = threadIdx.x & 31;
  const int rpb = p.box_rows;
  const uint8_t* ksb = reinterpret_cast<const uint8_t*>(p.k_scales);
  const uint8_t* vsb = reinterpret_cast<const uint8_t*>(p.v_scales);
  int page = box_page(p, pc, 0, lane);
  for (int jt = 0; jt < pc.n_tiles; ++jt) {
    const int next_page = box_page(p, pc, jt + 1, lane);
    const int gj = gj0 + jt;
    const int t0 = pc.tok_begin + jt * kTile;
    const int ntok = min(kTile, pc.tok_end - t0);
    const int nbox = (ntok + rpb - 1) / rpb;
    const int t = t0 + lane * rpb;
    const long long row =
        ((long long)(page * p.hkv + pc.g) << p.log2_ps) + (t & (p.page_size - 1));
    const uint32_t bytes = (uint32_t)(nbox * rpb * (2 * 128 + 8));
    const uint32_t o = lane * rpb;
#pragma unroll
    for (int kv = 0; kv < 2; ++kv) {  // the K bytes, then the V bytes
      const int S = kv ? kVStages : kKStages, st = gj % S;
      uint64_t* empty = kv ? cx.bars->v8_empty : cx.bars->k8_empty;
      uint64_t* fullb = kv ? cx.bars->v8_full : cx.bars->k8_full;
      const bool ok = gj < S || wait_bar(cx, &empty[st], ((gj / S) - 1) & 1);
      if (!__all_sync(0xffffffffu, ok && !*cx.abort)) return false;
      const uint32_t full = tc::smem_u32(&fullb[st]);
      if (lane == 0) tc::bar_arrive_expect_tx(full, bytes);
      __syncwarp();
      if (lane < nbox) {
        const uint32_t base = tc::smem_u32(smem + (kv ? kOffVR + st * kVSlot
                                                      : kOffKR + st * kKSlot));
        const CUtensorMap* tm = kv ? tm_v : tm_k;
        tc::tma_load_2d(base + o * 128, tm, full, 0, (int)row);
        tc::tma_load_2d(base + kHalf + o * 128, tm, full, 128, (int)row);
        bulk_copy(base + kOffKS + o * 8, (kv ? vsb : ksb) + row * 8, rpb * 8, full);
      }
      *(kv ? last_v : last_k) = gj;
    }
    page = next_page;
  }
  return true;
}

// ---- warps 6..9: FP8 -> fp16 into the TMEM operand tiles -------------------
// Four E4M3 bytes -> two f16x2 (bytes 0,1 and bytes 2,3), each multiplied
// by its scale pair: the hardware E4M3x2 -> f16x2 conversion on each 16-bit
// half of the word, then one fp16 multiply per pair.
__device__ __forceinline__ void e4m3x4_scaled(uint32_t w, uint32_t s01,
                                              uint32_t s23, uint32_t& lo,
                                              uint32_t& hi) {
  uint32_t a, b;
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n"
      " cvt.rn.f16x2.e4m3x2 %0, l;\n cvt.rn.f16x2.e4m3x2 %1, h;\n}"
      : "=r"(a), "=r"(b)
      : "r"(w));
  const __half2 x = __hmul2(*reinterpret_cast<const __half2*>(&a),
                            *reinterpret_cast<const __half2*>(&s01));
  const __half2 y = __hmul2(*reinterpret_cast<const __half2*>(&b),
                            *reinterpret_cast<const __half2*>(&s23));
  lo = *reinterpret_cast<const uint32_t*>(&x);
  hi = *reinterpret_cast<const uint32_t*>(&y);
}

// Two transposed 16 x 16 byte blocks (x2): matrix m's rows are addressed by
// lanes 16 m .. 16 m + 15.  Thread 4 g + j receives, per matrix, column g
// (d0) and column g + 8 (d1), each holding rows 4 j .. 4 j + 3.
__device__ __forceinline__ void ldsm_x2_trans_b8(uint32_t addr, uint32_t* d) {
  asm volatile(
      "ldmatrix.sync.aligned.m16n16.x2.trans.shared.b8 {%0, %1, %2, %3}, [%4];"
      : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
      : "r"(addr));
}

// Loads of one V^T conversion step `it` (slot half it / 4, channel half
// (it / 2) % 2, 16-channel group it % 2) for lane quarter q4: the four
// transposed 16 x 16 blocks of the slot half's 64 tokens (d[2 tb], d[2 tb+1]
// = channel g and g + 8 of tokens 16 tb + 4 j .. + 3) and their scale pairs
// (s[2 tb], s[2 tb + 1] = tokens 16 tb + 4 j + {0, 1} and + {2, 3}).
__device__ __forceinline__ void load_v_step(const uint8_t* vp, int it, int q4,
                                            int lane, int jq, uint32_t* d,
                                            uint32_t* s) {
  const int sub = it >> 2, h = (it >> 1) & 1, gi = it & 1;
  const int cg = 2 * q4 + gi;  // 16-byte chunk of the half row
  const uint8_t* vb = vp + h * kHalf;
  const uint16_t* vsc = reinterpret_cast<const uint16_t*>(
      vp + kOffVT + (2 * h + (q4 >> 1)) * (kTile * 2));
#pragma unroll
  for (int tb = 0; tb < 4; tb += 2) {
    const int T = kSub * sub + 16 * tb + lane;  // lanes 16..31: the next block
    uint32_t x[4];
    ldsm_x2_trans_b8(tc::smem_u32(vb + T * 128 + ((cg ^ (T & 7)) << 4)), x);
    d[2 * tb] = x[0];
    d[2 * tb + 1] = x[1];
    d[2 * tb + 2] = x[2];
    d[2 * tb + 3] = x[3];
  }
#pragma unroll
  for (int tb = 0; tb < 4; ++tb) {
    const uint2 p = *reinterpret_cast<const uint2*>(vsc + kSub * sub + 16 * tb +
                                                    4 * jq);
    s[2 * tb] = p.x;
    s[2 * tb + 1] = p.y;
  }
}

__device__ __forceinline__ uint32_t dup_half(uint32_t h16) {
  return (h16 & 0xFFFFu) | (h16 << 16);
}

template <int NR>
__device__ void dequant_piece(const Ctx& cx, const Piece& pc, int gj0,
                              uint8_t* smem, uint32_t tmem, int set,
                              uint32_t& vpar) {
  constexpr int VS = Cols<NR>::kVSlots;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q4 = warp & 3;              // TMEM lane quarter of this warp
  const int L = 32 * q4 + lane;         // token (K) or channel (V^T) lane
  const uint32_t lane_base = tmem + ((uint32_t)(32 * q4) << 16);
  const int jq = lane & 3;  // token quad of the transposed V blocks
  const int kswz = L & 7;

  // the two warp sets take alternate tiles (by global tile index)
  for (int jt = (set - gj0) & 1; jt < pc.n_tiles; jt += 2) {
    const int gj = gj0 + jt;
    const int t0 = pc.tok_begin + jt * kTile;
    const int ntok = min(kTile, pc.tok_end - t0);
    const int sk = gj % kKStages, sv = gj % kVStages;
    uint8_t* kp = smem + kOffKR + sk * kKSlot;
    uint8_t* vp = smem + kOffVR + sv * kVSlot;
    wait_bar(cx, &cx.bars->k8_full[sk], (gj / kKStages) & 1);

    // ---- K: token L -> lane L, in two halves of 128 channels (TMEM columns
    // 0..63 and 64..127).  The first half is free once the first eight MMAs
    // of S^T_{j-1} are done, the second once S^T_{j-1} is complete, so the
    // first half of this tile is written while S^T_{j-1} still runs.
    const bool has = 32 * q4 < ntok;  // warp-uniform; lanes past the tile
                                      // are masked by the softmax
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
      if (gj > 0) {
        if (half == 0)  // QK^T of tile gj-1, committed to this set's barrier
          wait_bar(cx, &cx.bars->k_free_a[gj & 1], ((gj - 1) >> 1) & 1);
        else
          wait_bar(cx, &cx.bars->s_full[(gj - 1) & 1], ((gj - 1) >> 1) & 1);
      }
      tc::fence_after();
      if (has) {
        // the half row (8 x 16 bytes) and its two scales, all in flight
        uint4 raw[8];
        uint32_t ksc[2];
        const uint32_t k2 =
            *reinterpret_cast<const uint32_t*>(kp + kOffKS + L * 8 + 4 * half);
        ksc[0] = dup_half(k2);
        ksc[1] = dup_half(k2 >> 16);
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
          raw[cc] = *reinterpret_cast<const uint4*>(
              kp + half * kHalf + L * 128 + ((cc ^ kswz) << 4));
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          uint32_t o[32];
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const uint4 r4 = raw[bb * 4 + cc];
            const uint32_t w[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              e4m3x4_scaled(w[e], ksc[bb], ksc[bb], o[cc * 8 + 2 * e],
                            o[cc * 8 + 2 * e + 1]);
          }
          tc::tmem_st_cols<32>(lane_base + kColK + (2 * half + bb) * 32, o);
        }
      }
      tc::tmem_wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0)
        tc::bar_arrive(tc::smem_u32(half ? &cx.bars->k_full : &cx.bars->k_full_a));
    }
    if (lane == 0) tc::bar_arrive(tc::smem_u32(&cx.bars->k8_empty[sk]));

    // V scales of token L, transposed to [block][token] for the V^T pass
    wait_bar(cx, &cx.bars->v8_full[sv], (gj / kVStages) & 1);
    {
      const uint2 v4 = *reinterpret_cast<const uint2*>(vp + kOffKS + L * 8);
      uint16_t* vt = reinterpret_cast<uint16_t*>(vp + kOffVT);
      vt[0 * kTile + L] = (uint16_t)(v4.x & 0xFFFFu);
      vt[1 * kTile + L] = (uint16_t)(v4.x >> 16);
      vt[2 * kTile + L] = (uint16_t)(v4.y & 0xFFFFu);
      vt[3 * kTile + L] = (uint16_t)(v4.y >> 16);
    }

    // ---- V^T, one 64-token slot at a time: 16 x 16 blocks (16 tokens x 16
    // channels) through the transposing matrix load: thread 4 g + j gets
    // channel g (and g + 8) of tokens 4 j .. 4 j + 3, which after the
    // conversion is the register layout of a 16-lane x 256-bit TMEM store
    // (lane = channel, column = token pair).  Warp q4 covers channels
    // 32 q4 .. 32 q4 + 31 of each half.  The transposed scales come from
    // all four warps.
    tc::bar_sync_named(3 + set, 128);
#pragma unroll 1
    for (int sub = 0; sub < 2; ++sub) {
      const int u = 2 * gj + sub, slot = u % VS;
      if (u >= VS) {
        // the slot's previous 64 tokens are through PV: this set's barrier
        // of the slot, whose next parity is bit `slot` of vpar
        wait_bar(cx, &cx.bars->v_empty[slot][set], (vpar >> slot) & 1u);
        vpar ^= 1u << slot;
      }
      tc::fence_after();
#pragma unroll 1
      for (int hg = 0; hg < 4; ++hg) {
        const int h = hg >> 1, gi = hg & 1;  // half, 16-channel group
        uint32_t d[8], sc[8];
        load_v_step(vp, 4 * sub + hg, q4, lane, jq, d, sc);
        uint32_t o[16];  // token block tb of the slot: o[4 tb .. 4 tb + 3]
#pragma unroll
        for (int tb = 0; tb < 4; ++tb) {
          e4m3x4_scaled(d[2 * tb], sc[2 * tb], sc[2 * tb + 1], o[4 * tb],
                        o[4 * tb + 1]);
          e4m3x4_scaled(d[2 * tb + 1], sc[2 * tb], sc[2 * tb + 1],
                        o[4 * tb + 2], o[4 * tb + 3]);
        }
        if (ntok < kTile) {  // tokens past the piece: zero (0 * NaN poisons PV)
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int tk = kSub * sub + 16 * (k >> 2) + 4 * jq + 2 * (k & 1);
            if (tk >= ntok) o[k] = 0u;
            else if (tk + 1 >= ntok) o[k] &= 0xFFFFu;
          }
        }
        tc::tmem_st_16x256b_x4(lane_base + ((uint32_t)(16 * gi) << 16) + kColV +
                                   slot * 64 + h * 32,
                               o);
      }
      tc::tmem_wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) tc::bar_arrive(tc::smem_u32(&cx.bars->v_full[slot]));
    }
    if (lane == 0) tc::bar_arrive(tc::smem_u32(&cx.bars->v8_empty[sv]));
  }
}

// ---- MMA issue: warp 1 issues S^T_j, warp 10 issues O^T += V^T_j P^T_j --------
// Two issuing threads, each waiting (bounded, without polling) for its own
// inputs in tile order, so a ready PV never waits behind a QK^T issue and
// the other way round.  A commit tracks the MMAs of its own thread.
template <int NR>
__device__ void qk_piece(const Ctx& cx, const Piece& pc, int gj0,
                         uint32_t tmem) {
  // kind::f16 with fp16 A and B, fp32 D, M = 128, N = NR, B K-major
  constexpr uint32_t kIdQK = (1u << 4) | ((uint32_t)(NR >> 3) << 17) |
                             ((uint32_t)(128 >> 4) << 24);
  const uint64_t qdesc = tc::desc_sw128(
      tc::smem_u32(reinterpret_cast<uint8_t*>(cx.smem) + kOffQ), 16, 1024);
  for (int jt = 0; jt < pc.n_tiles; ++jt) {
    const int gj = gj0 + jt;
    // first half of K (channels 0..127) written, and the S^T buffer of tile
    // gj free (softmax consumed tile gj-2)
    wait_bar(cx, &cx.bars->k_full_a, gj & 1);
    if (gj >= 2) wait_bar(cx, &cx.bars->p_full[gj & 1], ((gj >> 1) - 1) & 1);
    tc::fence_after();
    const uint32_t d = tmem + Cols<NR>::kS + (gj & 1) * NR;
    // descriptors as the base descriptor plus constant address steps
    // (address field = byte address / 16; every operand lies below 256 KB,
    // so the field never carries)
#pragma unroll
    for (int k = 0; k < 8; ++k)
      tc::mma_bf16_ta(d, tmem + kColK + k * 8,
                      qdesc + (uint64_t)(((k >> 2) * (NR * 128) + (k & 3) * 32) >> 4),
                      kIdQK, k > 0 ? 1u : 0u);
    // after those eight MMAs, to the barrier of tile gj+1's dequant set
    tc::commit(tc::smem_u32(&cx.bars->k_free_a[(gj + 1) & 1]));
    wait_bar(cx, &cx.bars->k_full, gj & 1);        // second half written
    tc::fence_after();
#pragma unroll
    for (int k = 8; k < 16; ++k)
      tc::mma_bf16_ta(d, tmem + kColK + k * 8,
                      qdesc + (uint64_t)(((k >> 2) * (NR * 128) + (k & 3) * 32) >> 4),
                      kIdQK, 1u);
    tc::commit(tc::smem_u32(&cx.bars->s_full[gj & 1]));
  }
}

template <int NR>
__device__ void pv_piece(const Ctx& cx, const Piece& pc, int gj0,
                         uint32_t tmem) {
  using C = Cols<NR>;
  // B = P^T is MN-major
  constexpr uint32_t kIdPV = (1u << 4) | (1u << 16) |
                             ((uint32_t)(NR >> 3) << 17) |
                             ((uint32_t)(128 >> 4) << 24);
  uint8_t* smem = reinterpret_cast<uint8_t*>(cx.smem);
  const uint64_t pdesc0 = tc::desc_sw128(tc::smem_u32(smem + kOffP), 8192, 1024);
  const uint64_t pdesc1 =
      tc::desc_sw128(tc::smem_u32(smem + kOffP + kPBytes), 8192, 1024);
  for (int jt = 0; jt < pc.n_tiles; ++jt) {
    const int gj = gj0 + jt;
    const int t0 = pc.tok_begin + jt * kTile;
    const int nk = (min(kTile, pc.tok_end - t0) + 15) >> 4;
    const uint64_t pdesc = (gj & 1) ? pdesc1 : pdesc0;
    wait_bar(cx, &cx.bars->p_full[gj & 1], (gj >> 1) & 1);
    // two halves of 64 tokens, each from its V^T slot, so a slot is
    // released as soon as its tokens are through
#pragma unroll 1
    for (int sub = 0; sub < 2; ++sub) {
      const int u = 2 * gj + sub, slot = u % C::kVSlots;
      wait_bar(cx, &cx.bars->v_full[slot], (u / C::kVSlots) & 1);
      tc::fence_after();
      const uint32_t acc0 = (jt > 0 || sub > 0) ? 1u : 0u;
      // the two channel halves accumulate into separate O^T tiles: their
      // MMAs alternate so that two independent chains are in flight
#pragma unroll
      for (int k = 0; k < kSub / 16; ++k) {
        if (4 * sub + k < nk) {
#pragma unroll
          for (int h = 0; h < 2; ++h)
            tc::mma_bf16_ta(
                tmem + C::kO + h * NR, tmem + kColV + slot * 64 + h * 32 + k * 8,
                pdesc + (uint64_t)(((4 * sub + k) * 2048) >> 4), kIdPV,
                k > 0 ? 1u : acc0);
        }
      }
      // the slot's next writer: occurrence u + VS, tile (u + VS) / 2
      tc::commit(tc::smem_u32(&cx.bars->v_empty[slot][((u + C::kVSlots) >> 1) & 1]));
    }
    tc::commit(tc::smem_u32(&cx.bars->pv_done[gj & 1]));
  }
}

// ---- warps 2..5: Q, softmax and epilogue -------------------------------------
// Q of the piece as the QK^T B operand: NR rows x 256 fp16 channels, four
// 64-channel column blocks of NR x 128 bytes, 128-byte swizzle; rows past
// the block are zeros.  Also the rows' causal limits and output offsets.
template <int NR>
__device__ void load_q(const AttnParams& p, const Piece& pc, uint8_t* smem,
                       Red* red, int slot, int S) {
  const int tid = threadIdx.x;  // softmax warps 0..3
  const int qb = block_rows(p, pc.b);
  constexpr int kPer = NR * 32 / 128;  // 16-byte chunks per thread
  uint4 x[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const int idx = tid + 128 * e, r = idx >> 5, ch = idx & 31;
    const int i = r / p.group;
    const bool ok = r < p.rows && i < qb;
    const int head = pc.g * p.group + (r - i * p.group);
    x[e] = ok ? __ldg(reinterpret_cast<const uint4*>(
                    p.q + (((long long)pc.b * p.q_len + i) * p.hq + head) *
                              kHeadDim + ch * 8))
              : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const int idx = tid + 128 * e, r = idx >> 5, ch = idx & 31;
    uint32_t* w = reinterpret_cast<uint32_t*>(&x[e]);
#pragma unroll
    for (int k = 0; k < 4; ++k) {  // bf16 pairs -> fp16 pairs
      const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&w[k]);
      const __half2 h2 = __floats2half2_rn(__low2float(b2), __high2float(b2));
      w[k] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    const int cb = ch >> 3, c16 = ch & 7;
    *reinterpret_cast<uint4*>(smem + kOffQ + cb * (NR * 128) + r * 128 +
                              ((c16 ^ (r & 7)) << 4)) = x[e];
  }
  if (tid < NR) {
    const int r = tid, i = r / p.group;
    const bool ok = r < p.rows && i < qb;
    red->lim[r] = ok ? causal_limit(pc.len, qb, i) : 0;
    const int head = pc.g * p.group + (r - i * p.group);
    red->out_off[r] =
        r >= p.rows ? -1LL
                    : (S == 1 ? (((long long)pc.b * p.q_len + i) * p.hq + head) * kHeadDim
                              : ((long long)slot * p.rows + r) * kHeadDim);
  }
  tc::fence_proxy_async_smem();
}

// 16 score columns of S^T_j for this token, masked: a token past the tile
// or past row r's causal limit scores -inf.
__device__ __forceinline__ void load_scores16(uint32_t taddr, int c0,
                                              bool masked, bool in, int t,
                                              const Red* red, float* v) {
  tc::tmem_ld_cols<16>(taddr, reinterpret_cast<uint32_t*>(v));
  if (masked) {
    const int4* lim4 = reinterpret_cast<const int4*>(red->lim + c0);
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4) {
      const int4 lm = lim4[k4];
      if (!in || t >= lm.x) v[4 * k4] = -INFINITY;
      if (!in || t >= lm.y) v[4 * k4 + 1] = -INFINITY;
      if (!in || t >= lm.z) v[4 * k4 + 2] = -INFINITY;
      if (!in || t >= lm.w) v[4 * k4 + 3] = -INFINITY;
    }
  }
}

// P^T_j = 2^(s - m) for this token: its row of the MN-major B operand, 16
// rows (two 16-byte chunks) at a time, with the base-2 maxima `mu` (-inf
// replaced by 0).  Returns whether a score passed its row's maximum by more
// than 2^8 (then P^T_j must be recomputed after raising it; the values
// written may be as large as inf meanwhile, and are never published).
template <int NR>
__device__ __forceinline__ bool write_p(uint32_t sbuf, bool masked, bool in,
                                        int t, const Red* red, const float* mu,
                                        float sl2, uint8_t* prow, int L) {
  const float4* mu4 = reinterpret_cast<const float4*>(mu);
  bool need = false;
#pragma unroll 1
  for (int c0 = 0; c0 < NR; c0 += 16) {
    float v[16];
    load_scores16(sbuf + c0, c0, masked, in, t, red, v);
    uint32_t pk[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float4 m = mu4[(c0 >> 2) + (e >> 1)];
      const float m0 = (e & 1) ? m.z : m.x, m1 = (e & 1) ? m.w : m.y;
      const float a0 = fmaf(v[2 * e], sl2, -m0);
      const float a1 = fmaf(v[2 * e + 1], sl2, -m1);
      need |= a0 > kRescaleLog2;
      need |= a1 > kRescaleLog2;
      const __half2 hh = __floats2half2_rn(exp2f(a0), exp2f(a1));
      pk[e] = *reinterpret_cast<const uint32_t*>(&hh);
    }
    const int n8 = c0 >> 3;
    *reinterpret_cast<uint4*>(prow + ((n8 ^ (L & 7)) << 4)) =
        make_uint4(pk[0], pk[1], pk[2], pk[3]);
    *reinterpret_cast<uint4*>(prow + (((n8 + 1) ^ (L & 7)) << 4)) =
        make_uint4(pk[4], pk[5], pk[6], pk[7]);
  }
  return need;
}

template <int NR>
__device__ void softmax_piece(const Ctx& cx, const Piece& pc, int gj0,
                              uint32_t tmem, uint8_t* smem, Red* red, int slot,
                              int S) {
  const AttnParams& p = *cx.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q4 = warp & 3;
  const int L = 32 * q4 + lane;
  const uint32_t lane_base = tmem + ((uint32_t)(32 * q4) << 16);
  const float sl2 = p.scale_log2;
  const int qb = block_rows(p, pc.b);
  const int lim0 = causal_limit(pc.len, qb, 0);  // the smallest row limit

  // This token's share of each row sum.  The scores are re-read from TMEM
  // in 16-column chunks by each pass rather than held in registers.
  float lp[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) lp[r] = 0.f;
  int mi = 0;
  for (int jt = 0; jt < pc.n_tiles; ++jt) {
    const int gj = gj0 + jt;
    const int t0 = pc.tok_begin + jt * kTile;
    const int ntok = min(kTile, pc.tok_end - t0);
    const uint32_t sbuf = lane_base + Cols<NR>::kS + (gj & 1) * NR;
    const bool masked = ntok < kTile || t0 + kTile > lim0;
    const bool in = L < ntok;
    const int t = t0 + L;
    wait_bar(cx, &cx.bars->s_full[gj & 1], (gj >> 1) & 1);
    tc::fence_after();
    // P^T_j goes to the buffer of tile gj, free once PV of tile gj-2 is done
    if (gj >= 2) wait_bar(cx, &cx.bars->pv_done[gj & 1], ((gj >> 1) - 1) & 1);
    uint8_t* prow = smem + kOffP + (gj & 1) * kPBytes + L * 128;
    // Past the piece's first tile, P^T_j is written at once with the running
    // maxima, and the same pass notes a score that passes its row's maximum
    // by more than 2^8; the four warps then vote.  Only then (rarely) is m
    // raised and P^T_j written again, so a tile costs one pass over S^T.
    // Nothing is published before the vote.
    bool raise = jt == 0;  // the piece's first tile sets m from its scores
    for (;;) {
      if (raise) {
#pragma unroll 1
        for (int c0 = 0; c0 < NR; c0 += 16) {
          float v[16];
          load_scores16(sbuf + c0, c0, masked, in, t, red, v);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
              v[k] = fmaxf(v[k], __shfl_xor_sync(0xffffffffu, v[k], o));
          }
          if (lane == 0) {
#pragma unroll
            for (int k = 0; k < 16; ++k) red->colmax[q4][c0 + k] = v[k];
          }
        }
        tc::bar_sync_named(2, 128);
        if (L < NR) {
          // scale > 0, so the max of the raw scores gives the max of the scaled
          const float cm = fmaxf(fmaxf(red->colmax[0][L], red->colmax[1][L]),
                                 fmaxf(red->colmax[2][L], red->colmax[3][L])) * sl2;
          const float mo = red->m[mi][L];
          float mn = mo, al = 1.f;
          if (jt == 0) {
            mn = cm;
          } else if (mo != -INFINITY && cm > mo + kRescaleLog2) {
            mn = cm;
            al = exp2f(mo - mn);
          }
          red->m[mi ^ 1][L] = mn;
          red->mu[mi ^ 1][L] = mn == -INFINITY ? 0.f : mn;
          red->alpha[L] = al;
        }
        tc::bar_sync_named(2, 128);
        mi ^= 1;
        if (jt > 0) {
#pragma unroll
          for (int r = 0; r < NR; ++r) lp[r] *= red->alpha[r];
          // O^T must be final for tile gj-1 before it is rescaled
          wait_bar(cx, &cx.bars->pv_done[(gj - 1) & 1], ((gj - 1) >> 1) & 1);
          tc::fence_after();
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
#pragma unroll 1
            for (int c0 = 0; c0 < NR; c0 += 16) {
              uint32_t o[16];
              const uint32_t ta = lane_base + Cols<NR>::kO + h * NR + c0;
              tc::tmem_ld_cols<16>(ta, o);
#pragma unroll
              for (int k = 0; k < 16; ++k)
                o[k] = __float_as_uint(__uint_as_float(o[k]) * red->alpha[c0 + k]);
              tc::tmem_st16(ta, o);
            }
          }
          tc::tmem_wait_st();
        }
      }
      const bool need =
          write_p<NR>(sbuf, masked, in, t, red, red->mu[mi], sl2, prow, L);
      if (raise) break;  // written with the raised maxima
      const bool any = __any_sync(0xffffffffu, need);
      if (lane == 0) red->flag[gj & 1][q4] = any ? 1 : 0;
      tc::bar_sync_named(2, 128);
      raise = (red->flag[gj & 1][0] | red->flag[gj & 1][1] |
               red->flag[gj & 1][2] | red->flag[gj & 1][3]) != 0;
      if (!raise) break;
    }
    // this token's share of the row sums, from the fp16 P^T row it wrote:
    // the same values the PV MMAs multiply
#pragma unroll
    for (int n8 = 0; n8 < NR / 8; ++n8) {
      const uint4 w4 =
          *reinterpret_cast<const uint4*>(prow + ((n8 ^ (L & 7)) << 4));
      const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f =
            __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
        lp[8 * n8 + 2 * k] += f.x;
        lp[8 * n8 + 2 * k + 1] += f.y;
      }
    }
    tc::fence_proxy_async_smem();
    tc::fence_before();
    __syncwarp();
    if (lane == 0) tc::bar_arrive(tc::smem_u32(&cx.bars->p_full[gj & 1]));
  }

  // epilogue: row sums over the tokens, then O = O^T / l
  const int gl = gj0 + pc.n_tiles - 1;
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    float v = lp[r];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) red->lsum_w[q4][r] = v;
  }
  tc::bar_sync_named(2, 128);
  if (L < NR) {
    const float l = (red->lsum_w[0][L] + red->lsum_w[1][L]) +
                    (red->lsum_w[2][L] + red->lsum_w[3][L]);
    red->lsum[L] = l;
    red->inv[L] = (red->lim[L] > 0 && l > 0.f) ? 1.f / l : 0.f;
  }
  tc::bar_sync_named(2, 128);
  wait_bar(cx, &cx.bars->pv_done[gl & 1], (gl >> 1) & 1);
  tc::fence_after();
  // O = O^T / l, one 128-channel half at a time, staged row-major in the
  // two P^T buffers (free: PV of the last tile is done) and written by
  // bulk stores of one row each, issued by thread r for row r, so the
  // softmax warps never wait on global stores.  The next writer of the
  // staging area (the other half, or the next piece's P^T) first waits
  // until those stores have read it.
  uint8_t* stage = smem + kOffP;
  const uint32_t esz = S == 1 ? 2u : 4u;
#pragma unroll 1
  for (int h = 0; h < 2; ++h) {  // channel L + 128 h of every row
    if (h == 1) {
      if (L < NR) bulk_store_wait<false>();
      tc::bar_sync_named(2, 128);
    }
#pragma unroll 1
    for (int c0 = 0; c0 < NR; c0 += 16) {
      uint32_t o[16];
      tc::tmem_ld_cols<16>(lane_base + Cols<NR>::kO + h * NR + c0, o);
      float inv[16];
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        const float4 f = reinterpret_cast<const float4*>(red->inv + c0)[k4];
        inv[4 * k4] = f.x; inv[4 * k4 + 1] = f.y;
        inv[4 * k4 + 2] = f.z; inv[4 * k4 + 3] = f.w;
      }
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float v = __uint_as_float(o[k]) * inv[k];
        if (S == 1)
          reinterpret_cast<__nv_bfloat16*>(stage)[(c0 + k) * 128 + L] =
              __float2bfloat16_rn(v);
        else
          reinterpret_cast<float*>(stage)[(c0 + k) * 128 + L] = v;
      }
    }
    tc::fence_proxy_async_smem();
    tc::bar_sync_named(2, 128);
    if (L < NR) {
      const long long off = red->out_off[L];
      if (off >= 0) {
        void* dst = S == 1 ? static_cast<void*>(p.out + off + 128 * h)
                           : static_cast<void*>(p.part_o + off + 128 * h);
        bulk_store(dst, tc::smem_u32(stage + L * 128 * esz), 128 * esz);
      }
    }
  }
  if (S > 1 && L < p.rows) {
    const float l = red->lsum[L];
    p.part_lse[(long long)slot * p.rows + L] =
        (red->lim[L] > 0 && l > 0.f) ? red->mu[mi][L] + log2f(l) : -INFINITY;
  }
  if (L < NR) bulk_store_wait<false>();  // the staging area is P^T again
  tc::bar_sync_named(2, 128);
}

template <int NR>
__global__ void __launch_bounds__(kThreads, 1)
    verify_split_fp8t_kernel(const AttnParams p,
                             const __grid_constant__ CUtensorMap tm_k,
                             const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  int* s_pre = reinterpret_cast<int*>(smem + kOffPre);
  Red* red = reinterpret_cast<Red*>(smem + kOffRed);
  __shared__ __align__(8) Bars bars;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the merge kernel may be scheduled now; it waits for this grid to finish
  tc_grid_launch_dependents();
  // launched as a programmatic dependent of the kernel before it on the
  // stream (it was scheduled while that one ran): every input and output
  // is touched only once that grid is complete
  tc_grid_dependency_wait();
  plan_prefix(p, s_pre);
  const Plan pl = make_plan(p, (long long)p.hkv * s_pre[p.batch]);
  const int c = blockIdx.x;
  if (c >= pl.P) return;  // uniform over the CTA, before any TMEM or barrier use

  if (tid == 0) {
    for (int s = 0; s < kKStages; ++s) {
      tc::bar_init(tc::smem_u32(&bars.k8_full[s]), 1);
      tc::bar_init(tc::smem_u32(&bars.k8_empty[s]), 4);
    }
    for (int s = 0; s < kVStages; ++s) {
      tc::bar_init(tc::smem_u32(&bars.v8_full[s]), 1);
      tc::bar_init(tc::smem_u32(&bars.v8_empty[s]), 4);
    }
    tc::bar_init(tc::smem_u32(&bars.k_full_a), 4);
    tc::bar_init(tc::smem_u32(&bars.k_full), 4);
    tc::bar_init(tc::smem_u32(&bars.k_free_a[0]), 1);
    tc::bar_init(tc::smem_u32(&bars.k_free_a[1]), 1);
    for (int s = 0; s < 3; ++s) {
      tc::bar_init(tc::smem_u32(&bars.v_full[s]), 4);
      tc::bar_init(tc::smem_u32(&bars.v_empty[s][0]), 1);
      tc::bar_init(tc::smem_u32(&bars.v_empty[s][1]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::bar_init(tc::smem_u32(&bars.s_full[s]), 1);
      tc::bar_init(tc::smem_u32(&bars.p_full[s]), 4);
      tc::bar_init(tc::smem_u32(&bars.pv_done[s]), 1);
    }
    tc::bar_init(tc::smem_u32(&bars.drain), 2);
    s_abort = 0;
    tc::bar_fence_init();
  }
  if (warp == kWarpQK) tc::tmem_alloc(tc::smem_u32(&s_tmem), kTmemCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = s_tmem;
  Ctx cx{&bars, &s_abort, &p, smem};

  long long u = chunk_start(pl, c);
  const long long u_end = chunk_start(pl, c + 1);
  int gj0 = 0;
  int last_k = -1, last_v = -1;  // last tiles whose K / V loads were issued
  bool producing = true;         // producer: cleared once it stopped issuing
  uint32_t vpar = 0;     // dequant warps: parities of their V^T-slot waits
  while (u < u_end) {
    Piece pc;
    pc.b = find_request(s_pre, p.batch, p.hkv, u);
    const int ntv = s_pre[pc.b + 1] - s_pre[pc.b];  // virtual units
    const long long rb = (long long)p.hkv * s_pre[pc.b];
    pc.g = (int)((u - rb) / ntv);
    const long long vs = rb + (long long)pc.g * ntv;
    const int j0v = (int)(u - vs);
    const int j1v = (int)(u_end - vs < ntv ? u_end - vs : ntv);
    u = vs + j1v;
    // real units of the piece; a range of phantom units only does nothing
    const int j0 = max(j0v - p.piece_cost, 0), j1 = max(j1v - p.piece_cost, 0);
    if (j1 <= j0) continue;  // the same decision in every warp
    pc.nt = ntv - p.piece_cost;
    pc.s0 = vs + p.piece_cost;  // the segment's first real unit
    pc.len = clamp_len(p.seq_lens[pc.b], p.max_tokens);
    pc.tok_begin = j0 * kUnit;
    pc.tok_end = min(j1 * kUnit, pc.len);
    pc.n_tiles = (pc.tok_end - pc.tok_begin + kTile - 1) / kTile;

    // The producer and the dequant warps run ahead across pieces, gated by
    // the ring and operand barriers; the MMA issuer and the softmax warps
    // meet around each piece, so Q is rewritten only after the previous
    // piece's last MMA and O^T is read before the next piece's first PV.
    if (warp == kWarpProducer) {
      if (producing)
        producing = produce(cx, pc, gj0, smem, &tm_k, &tm_v, &last_k, &last_v);
      __syncwarp();
    } else if (warp >= 4 && warp < 12) {
      dequant_piece<NR>(cx, pc, gj0, smem, tmem, (warp - 4) >> 2, vpar);
    } else if (warp < 4 || warp == kWarpQK || warp == kWarpPV) {
      int S = 0, slot = 0;
      if (warp < 4) {
        // where this piece's result goes
        S = seg_splits(pl, pc.s0, pc.nt);
        slot = S > 1 ? partial_slot(c, pc.b * p.hkv + pc.g) : 0;
        load_q<NR>(p, pc, smem, red, slot, S);
      }
      tc::fence_before();
      tc::bar_sync_named(1, kPieceThreads);
      tc::fence_after();
      if (warp == kWarpQK || warp == kWarpPV) {
        if (lane == 0) {
          if (warp == kWarpQK) qk_piece<NR>(cx, pc, gj0, tmem);
          else pv_piece<NR>(cx, pc, gj0, tmem);
        }
        __syncwarp();
      } else {
        softmax_piece<NR>(cx, pc, gj0, tmem, smem, red, slot, S);
      }
      tc::fence_before();
      tc::bar_sync_named(1, kPieceThreads);
      tc::fence_after();
    }
    gj0 += pc.n_tiles;
  }

  // teardown: no copy, bulk store or MMA may still be in flight
  if (warp < 4 && tid < kRowsMax) bulk_store_wait<true>();
  if (warp == kWarpProducer && lane == 0) {
    for (int gj = max(0, last_k - kKStages + 1); gj <= last_k; ++gj)
      wait_bar(cx, &bars.k8_full[gj % kKStages], (gj / kKStages) & 1, true);
    for (int gj = max(0, last_v - kVStages + 1); gj <= last_v; ++gj)
      wait_bar(cx, &bars.v8_full[gj % kVStages], (gj / kVStages) & 1, true);
  }
  if ((warp == kWarpQK || warp == kWarpPV) && lane == 0) {  // both issuers
    tc::commit(tc::smem_u32(&bars.drain));
    wait_bar(cx, &bars.drain, 0, true);
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == kWarpQK) tc::tmem_dealloc(tmem, kTmemCols);
}

template <int NR>
cudaError_t launch(const AttnParams& p, const CUtensorMap& tm_k,
                   const CUtensorMap& tm_v, cudaStream_t s) {
  // the shared-memory attribute was set by verify_split_fp8t_ctas_per_sm(),
  // which sizing the grid always runs first
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg =
      pdl_config(dim3(p.grid), dim3(kThreads), kSmem, s, attr);
  return cudaLaunchKernelEx(&cfg, verify_split_fp8t_kernel<NR>, p, tm_k, tm_v);
}

template <int NR>
bool set_smem() {
  return cudaFuncSetAttribute(verify_split_fp8t_kernel<NR>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmem) == cudaSuccess;
}

}  // namespace

cudaError_t launch_verify_split_fp8t(const AttnParams& p,
                                     const CUtensorMap& tm_k,
                                     const CUtensorMap& tm_v, cudaStream_t s) {
  const int nr = (p.rows + 15) / 16 * 16;
  switch (nr) {
    case 16: return launch<16>(p, tm_k, tm_v, s);
    case 32: return launch<32>(p, tm_k, tm_v, s);
    case 48: return launch<48>(p, tm_k, tm_v, s);
    case 64: return launch<64>(p, tm_k, tm_v, s);
    default: return cudaErrorInvalidValue;
  }
}

int verify_split_fp8t_ctas_per_sm() {
  if (!set_smem<16>() || !set_smem<32>() || !set_smem<48>() || !set_smem<64>())
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &n, verify_split_fp8t_kernel<48>, kThreads, kSmem) != cudaSuccess)
    return 0;
  return n < 1 ? 0 : 1;  // TMEM: one 512-column allocation per SM
}

}  // namespace specv
