// Split-KV paged GQA verify attention on the 5th-generation tensor cores
// (tcgen05 MMA with TMEM operands and accumulators, TMA / bulk-copy loads),
// for bf16 KV and for FP8-E4M3 KV with fp16 scales.
//
// One CTA per SM walks its contiguous run of 64-token units (the plan in
// common.cuh).  For every (request b, KV head g) piece of the run, all
// q_len x group query rows that read KV head g form the M = 128 rows of one
// MMA tile ("MTP and DFlash2 at long context on XPU", Part III: the query
// positions of a verify block folded into the head dimension, so every KV
// byte is read once).  Query row r sits at TMEM lane 32*(r / R) + r % R,
// R = ceil(rows / 4), which spreads the rows over the four TMEM lane
// quarters; the other lanes carry zero rows.
//
// Tensor memory (512 columns): O accumulator [0, 256), two S/P buffers of 64
// columns [256, 384), the Q tile as an MMA A operand [384, 512) (256 16-bit
// channels, two per column, even channel in the low half).
//
// Warp roles:
//   warp 0      producer (all 32 lanes, lane i owns box i of a tile: a run of
//               min(page_size, 64) tokens of one page; page ids prefetched
//               one tile ahead).  bf16: 2-D TMA boxes of 64 channels with the
//               128-byte swizzle straight into a 3-stage K/V ring, fetched
//               with an evict-first L2 policy.  FP8: 1-D
//               bulk copies of the page runs of K/V bytes and their scales
//               into a 2-stage staging ring.
//   warp 1      MMA issuer (one thread): S_j = Q K_j^T (16 MMAs, N = 64) into
//               an S buffer and O += P_j V_j (N = 256, V as an MN-major
//               operand, P from TMEM) into O, each as soon as its inputs are
//               ready.
//   warps 2..5  softmax: one thread per TMEM lane (query row).  Load S_j,
//               mask the block's causal tail, keep a running max m and sum l
//               in base 2, write P_j = 2^(s - m) back over S_j; rescale O in
//               TMEM only when m grows by more than 2^8; finally read O,
//               divide by l and write the bf16 output or an fp32 partial.
//               bf16 KV: P is stored as bf16 hi + lo parts and PV runs once
//               per part (one bf16 P carries a 2^-9 relative error per
//               weight, visible in the output when few keys are visible).
//   warps 6..9  (FP8 only) dequant: element c of a cached row becomes
//               fp16(e4m3(byte_c) * scale[c / 64]) in the swizzled K/V stage
//               ("Qwen3.8-27B-FP8" page, "Implemented execution path": FP8
//               E4M3 cache with per-token / per-KV-head FP16 scales over
//               64-channel blocks).  The FP8 path computes in fp16 (Q, the
//               dequantised K/V and P), which holds 11 significant bits.
//
// The tile width is set by the MMA issue rate: QK^T costs 16 instructions
// per tile whatever its width, so 64-token tiles halve the instructions per
// KV byte of 32-token tiles.
//
// Every wait is bounded (AttnParams::wait_cycles, about two seconds by
// default); a wait that runs out sets SPEC_STATUS_TIMEOUT in the status word
// (checked mode) and makes every later wait of the CTA return at once, so
// the kernel always finishes.  The producer then issues no further loads,
// and the teardown waits (with the long bound) for the loads and MMAs
// already issued before it frees tensor memory.
#include <cuda_fp8.h>

#include "common.cuh"
#include "spec_verify.h"
#include "tc_ptx.cuh"

namespace specv {
namespace {

constexpr int kT = 64;                        // tokens per tile
constexpr int kHalfBytes = 4 * kT * 128;      // K (or V) of one 16-bit stage
constexpr int kStageBytes = 2 * kHalfBytes;
constexpr int kPreBytes = ((kMaxBatch + 1) * 4 + 127) / 128 * 128;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 256;               // S/P buffers: columns 256, 320
constexpr uint32_t kColQ = 384;               // Q: columns 384..511
constexpr float kRescaleLog2 = 8.0f;          // rescale O when m grows > 2^8
// FP8 staging: K bytes, V bytes, K scales, V scales of one tile
constexpr int kS8K = 0;
constexpr int kS8V = kT * 256;
constexpr int kS8KS = 2 * kT * 256;
constexpr int kS8VS = kS8KS + kT * 8;
constexpr int kS8Bytes = kS8VS + kT * 8;

// bf16: K/V stage s at s * kStageBytes (K) and + kHalfBytes (V), one
// barrier pair per stage.  FP8: separate 2-slot K and V rings, so a K slot
// is refilled as soon as its QK^T is done rather than after the PV.
template <bool kFp8>
struct Cfg {
  static constexpr int kStages = kFp8 ? 2 : 3;
  static constexpr int kStages8 = kFp8 ? 2 : 0;
  static constexpr int kThreads = kFp8 ? 320 : 192;
  static constexpr int kOffKV = 0;
  static constexpr int kOff8 = kOffKV + kStages * kStageBytes;
  static constexpr int kOffPre = kOff8 + kStages8 * kS8Bytes;
  __device__ static uint32_t k_off(int gj) {
    return kFp8 ? (gj % kStages) * kHalfBytes : (gj % kStages) * kStageBytes;
  }
  __device__ static uint32_t v_off(int gj) {
    return kFp8 ? kStages * kHalfBytes + (gj % kStages) * kHalfBytes
                : (gj % kStages) * kStageBytes + kHalfBytes;
  }
  static constexpr int kSmem = kOffPre + kPreBytes + 1024;  // + alignment
  // kind::f16 with bf16 (1) or fp16 (0) inputs, fp32 accumulator
  static constexpr uint32_t kAB = kFp8 ? 0u : 1u;
  static constexpr uint32_t kIdescQK = (1u << 4) | (kAB << 7) | (kAB << 10) |
                                       ((uint32_t)(kT >> 3) << 17) |
                                       ((uint32_t)(128 >> 4) << 24);
  static constexpr uint32_t kIdescPV = (1u << 4) | (kAB << 7) | (kAB << 10) |
                                       (1u << 16) | ((uint32_t)(256 >> 3) << 17) |
                                       ((uint32_t)(128 >> 4) << 24);
};

struct Bars {
  uint64_t kv_full[3];    // bf16: stage holds tile j (TMA tx); FP8: K slot
  uint64_t kv_empty[3];   // bf16: PV of the stage's tile done; FP8: QK done
  uint64_t v_full[2];     // FP8: V slot dequantised
  uint64_t v_empty[2];    // FP8: PV of the V slot's tile done
  uint64_t f8_full[2];    // FP8 staging landed (bulk-copy tx)
  uint64_t f8_empty[2];   // dequant consumed the staging buffer
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t pv_done[2];
  uint64_t drain;
};

struct Ctx {
  Bars* bars;
  volatile int* abort;
  const AttnParams* p;
};

// Bounded wait on phase `parity` of an mbarrier.  Returns false (and flags
// the CTA) when the bound runs out or another wait of the CTA already did.
// The teardown's drain (ignore_abort) keeps the long bound whatever the
// main-loop bound is: copies and MMAs already issued must land before the
// CTA frees its tensor memory and exits.
__device__ __noinline__ bool wait_slow(uint32_t a, uint32_t parity,
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

struct Piece {
  int b, g, nt, len, tok_begin, tok_end, n_tiles;
  long long s0;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src,
                                          uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// The KV tiles are read once: they are fetched with an L2 policy that makes
// their lines the first to be evicted, so the stream neither pushes other
// data out of L2 nor, after a write-heavy kernel, makes L2 write back its
// dirty lines ahead of the reads (measured: 0.839 -> 0.871 of the copy
// bandwidth on a 1 GB call after a 512 MB write, 0.888 -> 0.902 back to
// back on 8 x 32K tokens; the FP8 kernel measured slower with it).
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;"
               : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void tma_load_2d_evict_first(uint32_t dst,
                                                        const CUtensorMap* map,
                                                        uint32_t bar, int x,
                                                        int y, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_"
      "tx::bytes.L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(pol)
      : "memory");
}

// ---- warp 0: loads of the piece's K/V tiles ---------------------------------
__device__ __forceinline__ int box_page(const AttnParams& p, const Piece& pc,
                                        int jt, int lane) {
  const int t = pc.tok_begin + jt * kT + lane * p.box_rows;
  if (jt >= pc.n_tiles || t >= pc.tok_end || lane * p.box_rows >= kT) return 0;
  int page = __ldg(p.page_table + (long long)pc.b * p.max_pages +
                   (t >> p.log2_ps));
  if (page < 0 || page >= p.num_pages) {
    if (p.status) atomicOr(p.status, SPEC_STATUS_BAD_PAGE);
    page = 0;  // in bounds; the affected rows are unspecified
  }
  return page;
}

// Returns the number of tiles whose loads were issued: all of the piece's,
// unless the CTA gave up (a wait ran out), after which nothing more is
// issued, so that the teardown can wait for exactly the loads in flight.
// A stage is refilled only once its previous tile's data has landed and
// been consumed, so at most one load per stage is ever in flight.
template <bool kFp8>
__device__ int produce(const Ctx& cx, const Piece& pc, int gj0, uint8_t* smem,
                       const CUtensorMap* tm_k, const CUtensorMap* tm_v) {
  using C = Cfg<kFp8>;
  const AttnParams& p = *cx.p;
  const int lane = threadIdx.x & 31;
  const int rpb = p.box_rows;
  const uint64_t pol = l2_evict_first();
  int page = box_page(p, pc, 0, lane);
  for (int jt = 0; jt < pc.n_tiles; ++jt) {
    const int next_page = box_page(p, pc, jt + 1, lane);
    const int gj = gj0 + jt;
    const int t0 = pc.tok_begin + jt * kT;
    const int ntok = min(kT, pc.tok_end - t0);
    const int nbox = (ntok + rpb - 1) / rpb;
    const int t = t0 + lane * rpb;
    // row of this box's first token in the [num_pages * Hkv * page_size] view
    const long long row =
        ((long long)(page * p.hkv + pc.g) << p.log2_ps) + (t & (p.page_size - 1));
    if constexpr (!kFp8) {
      const int st = gj % C::kStages;
      bool ok = gj < C::kStages ||
                wait_bar(cx, &cx.bars->kv_empty[st], ((gj / C::kStages) - 1) & 1);
      if (!__all_sync(0xffffffffu, ok && !*cx.abort)) return jt;
      const uint32_t full = tc::smem_u32(&cx.bars->kv_full[st]);
      if (lane == 0)
        tc::bar_arrive_expect_tx(full, (uint32_t)(nbox * rpb * 128 * 4 * 2));
      __syncwarp();
      if (lane < nbox) {
        const uint32_t kdst = tc::smem_u32(smem + C::kOffKV + st * kStageBytes);
        const uint32_t vdst = kdst + kHalfBytes;
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
          const uint32_t off = cb * (kT * 128) + lane * rpb * 128;
          tma_load_2d_evict_first(kdst + off, tm_k, full, cb * 64, (int)row, pol);
          tma_load_2d_evict_first(vdst + off, tm_v, full, cb * 64, (int)row, pol);
        }
      }
    } else {
      const int s8 = gj % C::kStages8;
      bool ok = gj < C::kStages8 ||
                wait_bar(cx, &cx.bars->f8_empty[s8], ((gj / C::kStages8) - 1) & 1);
      if (!__all_sync(0xffffffffu, ok && !*cx.abort)) return jt;
      const uint32_t full = tc::smem_u32(&cx.bars->f8_full[s8]);
      if (lane == 0)
        tc::bar_arrive_expect_tx(full, (uint32_t)(nbox * rpb * (2 * 256 + 2 * 8)));
      __syncwarp();
      if (lane < nbox) {
        const uint32_t base = tc::smem_u32(smem + C::kOff8 + s8 * kS8Bytes);
        const uint8_t* kb = static_cast<const uint8_t*>(p.k_pages);
        const uint8_t* vb = static_cast<const uint8_t*>(p.v_pages);
        const uint8_t* ksb = reinterpret_cast<const uint8_t*>(p.k_scales);
        const uint8_t* vsb = reinterpret_cast<const uint8_t*>(p.v_scales);
        const uint32_t o = lane * rpb;
        bulk_copy(base + kS8K + o * 256, kb + row * 256, rpb * 256, full);
        bulk_copy(base + kS8V + o * 256, vb + row * 256, rpb * 256, full);
        bulk_copy(base + kS8KS + o * 8, ksb + row * 8, rpb * 8, full);
        bulk_copy(base + kS8VS + o * 8, vsb + row * 8, rpb * 8, full);
      }
    }
    page = next_page;
  }
  return pc.n_tiles;
}

// ---- warps 6..9 (FP8): dequantise a staged tile into the fp16 K/V slots -----
// Thread t converts 16-byte input chunks c16 = t & 15 of rows (t >> 4) + 8k
// (k = 0..7), first of K, then of V: 16 E4M3 bytes = channels 16*c16 ..
// 16*c16+15, one 64-channel block and one scale, two 16-byte output chunks.
// A thread's rows agree modulo 8, so its swizzled output offsets and its
// scale offsets are fixed strides of k, and all eight loads of a half are
// issued before the first conversion.  Rows past the piece's last token are
// written as zeros (their bytes are not data).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t pair16, __half2 sc) {
  const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(
      static_cast<__nv_fp8x2_storage_t>(pair16), __NV_E4M3);
  const __half2 h = __hmul2(*reinterpret_cast<const __half2*>(&hr), sc);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ void dequant_piece(const Ctx& cx, const Piece& pc, int gj0,
                              uint8_t* smem) {
  using C = Cfg<true>;
  const int tid = threadIdx.x - 192;  // 0..127
  const int lane = threadIdx.x & 31;
  const int c16 = tid & 15, r0 = tid >> 4;  // rows r0 + 8k
  const int cb = c16 >> 2, ch0 = (c16 & 3) * 2;
  const int src_off = r0 * 256 + c16 * 16;
  const int sc_off = r0 * 8 + cb * 2;
  const int dst_off0 = cb * (kT * 128) + r0 * 128 + ((ch0 ^ (r0 & 7)) << 4);
  const int dst_off1 = cb * (kT * 128) + r0 * 128 + (((ch0 + 1) ^ (r0 & 7)) << 4);
  for (int jt = 0; jt < pc.n_tiles; ++jt) {
    const int gj = gj0 + jt;
    const int s8 = gj % C::kStages8, st = gj % C::kStages;
    const int t0 = pc.tok_begin + jt * kT;
    const int nvalid = min(kT, pc.tok_end - t0);
    wait_bar(cx, &cx.bars->f8_full[s8], (gj / C::kStages8) & 1);
    const uint8_t* s8p = smem + C::kOff8 + s8 * kS8Bytes;
#pragma unroll
    for (int half = 0; half < 2; ++half) {  // K then V
      if (gj >= C::kStages)  // the slot's previous tile is done with it
        wait_bar(cx, half ? &cx.bars->v_empty[st] : &cx.bars->kv_empty[st],
                 ((gj / C::kStages) - 1) & 1);
      const uint8_t* src = s8p + (half ? kS8V : kS8K) + src_off;
      const uint8_t* scl = s8p + (half ? kS8VS : kS8KS) + sc_off;
      uint8_t* out = smem + (half ? C::v_off(gj) : C::k_off(gj));
      uint4 raw[8];
      __half sc[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        raw[k] = *reinterpret_cast<const uint4*>(src + k * 8 * 256);
        sc[k] = *reinterpret_cast<const __half*>(scl + k * 8 * 8);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const __half2 s2 = __halves2half2(sc[k], sc[k]);
        const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
        uint4 a, b;
        a.x = e4m3x2_to_f16x2(w[0] & 0xFFFF, s2);
        a.y = e4m3x2_to_f16x2(w[0] >> 16, s2);
        a.z = e4m3x2_to_f16x2(w[1] & 0xFFFF, s2);
        a.w = e4m3x2_to_f16x2(w[1] >> 16, s2);
        b.x = e4m3x2_to_f16x2(w[2] & 0xFFFF, s2);
        b.y = e4m3x2_to_f16x2(w[2] >> 16, s2);
        b.z = e4m3x2_to_f16x2(w[3] & 0xFFFF, s2);
        b.w = e4m3x2_to_f16x2(w[3] >> 16, s2);
        if (r0 + 8 * k >= nvalid) {
          a = make_uint4(0, 0, 0, 0);
          b = a;
        }
        *reinterpret_cast<uint4*>(out + dst_off0 + k * 8 * 128) = a;
        *reinterpret_cast<uint4*>(out + dst_off1 + k * 8 * 128) = b;
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0)
        tc::bar_arrive(tc::smem_u32(half ? &cx.bars->v_full[st]
                                         : &cx.bars->kv_full[st]));
    }
    if (lane == 0) tc::bar_arrive(tc::smem_u32(&cx.bars->f8_empty[s8]));
  }
}

// ---- warp 1, one thread: MMA issue -------------------------------------------
template <bool kFp8>
__device__ __forceinline__ void issue_qk(const Ctx& cx, int gj, uint32_t tmem,
                                         uint8_t* smem) {
  using C = Cfg<kFp8>;
  const uint32_t kbase = tc::smem_u32(smem + C::k_off(gj));
  const uint32_t d = tmem + kColS + (gj & 1) * kT;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const uint64_t bd = tc::desc_sw128(kbase + (k >> 2) * (kT * 128) + (k & 3) * 32, 16, 1024);
    tc::mma_bf16_ta(d, tmem + kColQ + k * 8, bd, C::kIdescQK, k > 0 ? 1u : 0u);
  }
  if (kFp8) tc::commit(tc::smem_u32(&cx.bars->kv_empty[gj % C::kStages]));
  tc::commit(tc::smem_u32(&cx.bars->s_full[gj & 1]));
}

template <bool kFp8>
__device__ __forceinline__ void issue_pv(const Ctx& cx, int gj, bool first,
                                         uint32_t tmem, uint8_t* smem) {
  using C = Cfg<kFp8>;
  const int st = gj % C::kStages;
  const uint32_t vbase = tc::smem_u32(smem + C::v_off(gj));
  const uint32_t p_hi = tmem + kColS + (gj & 1) * kT;  // 32 columns: pairs
  const uint32_t p_lo = p_hi + kT / 2;
#pragma unroll
  for (int kk = 0; kk < kT / 16; ++kk) {
    const uint64_t bd = tc::desc_sw128(vbase + kk * 2048, kT * 128, 1024);
    tc::mma_bf16_ta(tmem, p_hi + kk * 8, bd, C::kIdescPV,
                    (first && kk == 0) ? 0u : 1u);
    if (!kFp8) tc::mma_bf16_ta(tmem, p_lo + kk * 8, bd, C::kIdescPV, 1u);
  }
  tc::commit(tc::smem_u32(kFp8 ? &cx.bars->v_empty[st] : &cx.bars->kv_empty[st]));
  tc::commit(tc::smem_u32(&cx.bars->pv_done[gj & 1]));
}

template <bool kFp8>
__device__ void mma_piece(const Ctx& cx, const Piece& pc, int gj0, uint32_t tmem,
                          uint8_t* smem) {
  using C = Cfg<kFp8>;
  int qk = 0, pv = 0;
  long long last = clock64();
  while (pv < pc.n_tiles) {
    bool did = false;
    if (qk < pc.n_tiles) {
      const int gj = gj0 + qk;
      // the S/P buffer of tile gj is free once PV of tile gj-2 is done
      if (tc::bar_test_wait(tc::smem_u32(&cx.bars->kv_full[gj % C::kStages]),
                           (gj / C::kStages) & 1) &&
          (gj < 2 || tc::bar_test_wait(tc::smem_u32(&cx.bars->pv_done[gj & 1]),
                                      ((gj >> 1) - 1) & 1))) {
        tc::fence_after();
        issue_qk<kFp8>(cx, gj, tmem, smem);
        ++qk;
        did = true;
      }
    }
    if (pv < qk) {
      const int gj = gj0 + pv;
      if (tc::bar_test_wait(tc::smem_u32(&cx.bars->p_full[gj & 1]),
                           (gj >> 1) & 1) &&
          (!kFp8 || tc::bar_test_wait(tc::smem_u32(&cx.bars->v_full[gj % C::kStages]),
                                     (gj / C::kStages) & 1))) {
        tc::fence_after();
        issue_pv<kFp8>(cx, gj, pv == 0, tmem, smem);
        ++pv;
        did = true;
      }
    }
    if (did) {
      last = clock64();
    } else if (*cx.abort) {
      break;
    } else if (clock64() - last > cx.p->wait_cycles) {
      *cx.abort = 1;
      if (cx.p->status) atomicOr(cx.p->status, SPEC_STATUS_TIMEOUT);
      break;
    }
  }
}

// ---- warps 2..5: Q load, softmax and epilogue -------------------------------
// Each softmax thread writes its TMEM lane of the Q operand: the query row it
// owns (bf16, or converted to fp16 for FP8 KV), or zeros.
template <bool kFp8>
__device__ __forceinline__ void load_q_tmem(const AttnParams& p, const Piece& pc,
                                            uint32_t tmem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int w4 = warp & 3;
  const int R = (p.rows + 3) >> 2;
  const int r = w4 * R + lane;
  const bool in_tile = lane < R && r < p.rows;
  const int i = in_tile ? r / p.group : 0;
  const int h = pc.g * p.group + (in_tile ? r - i * p.group : 0);
  // rows past the request's block are never read (they may hold anything)
  const bool valid = in_tile && i < block_rows(p, pc.b);
  const uint4* src = reinterpret_cast<const uint4*>(
      p.q + (((long long)pc.b * p.q_len + i) * p.hq + h) * kHeadDim);
  const uint32_t lane_base = tmem + ((uint32_t)(32 * w4) << 16) + kColQ;
  uint4 xs[32];  // the whole row: every load in flight at once
#pragma unroll
  for (int k = 0; k < 32; ++k)
    xs[k] = valid ? __ldg(src + k) : make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
#pragma unroll
    for (int cq = 0; cq < 2; ++cq) {  // 64 channels = 32 columns per store
      const int cb = half * 2 + cq;
      uint32_t v[32];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        uint4 x = xs[half * 16 + cq * 8 + k];
        if (kFp8) {  // bf16 pairs -> fp16 pairs
          uint32_t* w = reinterpret_cast<uint32_t*>(&x);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&w[e]);
            const __half2 h2 = __floats2half2_rn(__low2float(b2), __high2float(b2));
            w[e] = *reinterpret_cast<const uint32_t*>(&h2);
          }
        }
        v[4 * k] = x.x;
        v[4 * k + 1] = x.y;
        v[4 * k + 2] = x.z;
        v[4 * k + 3] = x.w;
      }
      tc::tmem_st32(lane_base + cb * 32, reinterpret_cast<const float*>(v));
    }
  }
  tc::tmem_wait_st();
}

template <bool kFp8>
__device__ void softmax_piece(const Ctx& cx, const Piece& pc, int gj0,
                              uint32_t tmem, uint8_t* smem,
                              const Plan& pl, int c) {
  using C = Cfg<kFp8>;
  const AttnParams& p = *cx.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int w4 = warp & 3;
  const int R = (p.rows + 3) >> 2;
  const int r = w4 * R + lane;
  const bool valid = lane < R && r < p.rows;
  const int i = valid ? r / p.group : 0;
  const int lim = causal_limit(pc.len, block_rows(p, pc.b), i);
  const uint32_t lane_base = tmem + ((uint32_t)(32 * w4) << 16);
  const float sl2 = p.scale_log2;
  // where this piece's result goes
  const int S = seg_splits(pl, pc.s0, pc.nt);
  const int slot = S > 1 ? partial_slot(c, pc.b * p.hkv + pc.g) : 0;

  float m = -INFINITY, l = 0.f;
  for (int jt = 0; jt < pc.n_tiles; ++jt) {
    const int gj = gj0 + jt;
    const uint32_t sbuf = lane_base + kColS + (gj & 1) * kT;
    wait_bar(cx, &cx.bars->s_full[gj & 1], (gj >> 1) & 1);
    tc::fence_after();
    float s[kT];
    tc::tmem_ld32(sbuf, s);
    tc::tmem_ld32(sbuf + 32, s + 32);

    const int t0 = pc.tok_begin + jt * kT;
    if (t0 + kT > lim) {  // the causal tail of the block reaches this tile
#pragma unroll
      for (int k = 0; k < kT; ++k)
        if (t0 + k >= lim) s[k] = -INFINITY;
    }
    float mx4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
    for (int k = 4; k < kT; ++k) mx4[k & 3] = fmaxf(mx4[k & 3], s[k]);
    // scale > 0, so the max of the raw scores gives the max of the scaled
    const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * sl2;
    bool need = false;
    float alpha = 1.f;
    if (jt == 0) {
      m = mx;
    } else if (m != -INFINITY) {
      const float mn = fmaxf(m, mx);
      if (mn > m + kRescaleLog2) {
        need = true;
        alpha = exp2f(m - mn);
        m = mn;
      }
    }
    if (__any_sync(0xffffffffu, need)) {
      // O must be final for tile gj-1 before it is rescaled
      wait_bar(cx, &cx.bars->pv_done[(gj - 1) & 1], ((gj - 1) >> 1) & 1);
      tc::fence_after();
#pragma unroll 1
      for (int cb = 0; cb < 8; ++cb) {
        float o[32];
        tc::tmem_ld32(lane_base + cb * 32, o);
#pragma unroll
        for (int k = 0; k < 32; ++k) o[k] *= alpha;
        tc::tmem_st32(lane_base + cb * 32, o);
      }
      tc::tmem_wait_st();
      l *= alpha;
    }
    const float mu = m == -INFINITY ? 0.f : m;
    float sum4[4] = {0.f, 0.f, 0.f, 0.f};
    uint32_t hi[kT / 2], lo[kT / 2];
#pragma unroll
    for (int k = 0; k < kT; k += 2) {
      const float x0 = exp2f(fmaf(s[k], sl2, -mu));
      const float x1 = exp2f(fmaf(s[k + 1], sl2, -mu));
      sum4[k & 3] += x0;
      sum4[(k & 3) + 1] += x1;
      if (kFp8) {
        const __half2 hh = __floats2half2_rn(x0, x1);
        hi[k >> 1] = *reinterpret_cast<const uint32_t*>(&hh);
      } else {
        const __nv_bfloat162 hh = __floats2bfloat162_rn(x0, x1);
        const __nv_bfloat162 ll =
            __floats2bfloat162_rn(x0 - __low2float(hh), x1 - __high2float(hh));
        hi[k >> 1] = *reinterpret_cast<const uint32_t*>(&hh);
        lo[k >> 1] = *reinterpret_cast<const uint32_t*>(&ll);
      }
    }
    l += (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
    // bf16: V rows past the piece's last token must be zero (0 * NaN
    // poisons PV); the FP8 dequant warps write those rows as zeros.
    if (!kFp8 && t0 + kT > pc.tok_end) {
      const int st = gj % C::kStages;
      wait_bar(cx, &cx.bars->kv_full[st], (gj / C::kStages) & 1);
      uint8_t* v = smem + C::v_off(gj);
      const int z0 = pc.tok_end - t0;
      const int n = (kT - z0) * 4 * 8;  // rows x column blocks x chunks
      for (int e = threadIdx.x - 64; e < n; e += 128) {
        const int row = z0 + e / 32, rem = e % 32, cb = rem >> 3, ch = rem & 7;
        *reinterpret_cast<uint4*>(v + cb * (kT * 128) + row * 128 + (ch << 4)) =
            make_uint4(0, 0, 0, 0);
      }
      tc::fence_proxy_async_smem();
    }
    // P_j over S_j: hi in the first 32 columns, lo (bf16) in the next 32
    tc::tmem_st32(sbuf, reinterpret_cast<const float*>(hi));
    if (!kFp8) tc::tmem_st32(sbuf + kT / 2, reinterpret_cast<const float*>(lo));
    tc::tmem_wait_st();
    tc::fence_before();
    __syncwarp();
    if (lane == 0) tc::bar_arrive(tc::smem_u32(&cx.bars->p_full[gj & 1]));
  }

  // epilogue: O / l
  const int gl = gj0 + pc.n_tiles - 1;
  wait_bar(cx, &cx.bars->pv_done[gl & 1], (gl >> 1) & 1);
  tc::fence_after();
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const float mu = m == -INFINITY ? 0.f : m;
  const int head = pc.g * p.group + (r - i * p.group);
  if (S == 1) {
    __nv_bfloat16* dst =
        p.out + (((long long)pc.b * p.q_len + i) * p.hq + head) * kHeadDim;
#pragma unroll 1
    for (int cb = 0; cb < 8; cb += 2) {  // 64 columns per TMEM load
      float o[64];
      tc::tmem_ld64(lane_base + cb * 32, o);
      if (valid) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          uint4 v;
          __nv_bfloat162 t;
          t = __floats2bfloat162_rn(o[8 * k] * inv, o[8 * k + 1] * inv);
          v.x = *reinterpret_cast<uint32_t*>(&t);
          t = __floats2bfloat162_rn(o[8 * k + 2] * inv, o[8 * k + 3] * inv);
          v.y = *reinterpret_cast<uint32_t*>(&t);
          t = __floats2bfloat162_rn(o[8 * k + 4] * inv, o[8 * k + 5] * inv);
          v.z = *reinterpret_cast<uint32_t*>(&t);
          t = __floats2bfloat162_rn(o[8 * k + 6] * inv, o[8 * k + 7] * inv);
          v.w = *reinterpret_cast<uint32_t*>(&t);
          *reinterpret_cast<uint4*>(dst + cb * 32 + 8 * k) = v;
        }
      }
    }
  } else {
    float* dst = p.part_o + ((long long)slot * p.rows + r) * kHeadDim;
#pragma unroll 1
    for (int cb = 0; cb < 8; cb += 2) {  // 64 columns per TMEM load
      float o[64];
      tc::tmem_ld64(lane_base + cb * 32, o);
      if (valid) {
#pragma unroll
        for (int k4 = 0; k4 < 16; ++k4)
          *reinterpret_cast<float4*>(dst + cb * 32 + 4 * k4) =
              make_float4(o[4 * k4] * inv, o[4 * k4 + 1] * inv,
                          o[4 * k4 + 2] * inv, o[4 * k4 + 3] * inv);
      }
    }
    if (valid)
      p.part_lse[(long long)slot * p.rows + r] =
          l > 0.f ? mu + log2f(l) : -INFINITY;
  }
}

constexpr int kPieceThreads = 5 * 32;  // warps 1..5: MMA issuer + softmax

template <bool kFp8>
__global__ void __launch_bounds__(Cfg<kFp8>::kThreads, 1)
    verify_split_tc_kernel(const AttnParams p,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v) {
  using C = Cfg<kFp8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  int* s_pre = reinterpret_cast<int*>(smem + C::kOffPre);
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
  const int c = blockIdx.x;  // this kernel runs static plans only
  if (c >= pl.P) return;  // uniform over the CTA, before any TMEM or barrier use

  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      // bf16: one arrival (the producer's expect_tx) plus the TMA bytes;
      // FP8: one arrival per dequant warp
      tc::bar_init(tc::smem_u32(&bars.kv_full[s]), kFp8 ? 4 : 1);
      tc::bar_init(tc::smem_u32(&bars.kv_empty[s]), 1);
      if (kFp8) {
        tc::bar_init(tc::smem_u32(&bars.v_full[s]), 4);
        tc::bar_init(tc::smem_u32(&bars.v_empty[s]), 1);
      }
    }
    for (int s = 0; s < C::kStages8; ++s) {
      tc::bar_init(tc::smem_u32(&bars.f8_full[s]), 1);
      tc::bar_init(tc::smem_u32(&bars.f8_empty[s]), 4);
    }
    for (int s = 0; s < 2; ++s) {
      tc::bar_init(tc::smem_u32(&bars.s_full[s]), 1);
      tc::bar_init(tc::smem_u32(&bars.p_full[s]), 4);
      tc::bar_init(tc::smem_u32(&bars.pv_done[s]), 1);
    }
    tc::bar_init(tc::smem_u32(&bars.drain), 1);
    s_abort = 0;
    tc::bar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc(tc::smem_u32(&s_tmem), kTmemCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = s_tmem;
  Ctx cx{&bars, &s_abort, &p};

  long long u = chunk_start(pl, c);
  const long long u_end = chunk_start(pl, c + 1);
  int gj0 = 0;
  int last_loaded = -1;  // last tile index the producer loaded
  bool producing = true;  // producer: cleared once it stopped issuing
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
    pc.n_tiles = (pc.tok_end - pc.tok_begin + kT - 1) / kT;

    // The producer (warp 0) and the FP8 dequant warps run ahead across
    // pieces, gated only by the ring barriers; the MMA issuer and the
    // softmax warps (1..5) meet around each piece, so Q in TMEM is written
    // after the previous piece's last MMA and read after it is complete.
    if (warp == 0) {
      // the whole warp: lanes issue the copies of their pages
      if (producing) {
        const int n = produce<kFp8>(cx, pc, gj0, smem, &tm_k, &tm_v);
        if (n > 0) last_loaded = gj0 + n - 1;
        producing = n == pc.n_tiles;
      }
      __syncwarp();
    } else if (warp >= 6) {
      if (kFp8) dequant_piece(cx, pc, gj0, smem);
    } else {
      if (warp >= 2) load_q_tmem<kFp8>(p, pc, tmem);
      tc::fence_before();
      tc::bar_sync_named(1, kPieceThreads);
      tc::fence_after();
      if (warp == 1) {
        if (lane == 0) mma_piece<kFp8>(cx, pc, gj0, tmem, smem);
        __syncwarp();
      } else {
        softmax_piece<kFp8>(cx, pc, gj0, tmem, smem, pl, c);
      }
      tc::fence_before();
      tc::bar_sync_named(1, kPieceThreads);
      tc::fence_after();
    }
    gj0 += pc.n_tiles;
  }

  // teardown: no copy or MMA may still be in flight
  if (warp == 0 && lane == 0) {
    const int S = kFp8 ? C::kStages8 : C::kStages;
    for (int gj = max(0, last_loaded - S + 1); gj <= last_loaded; ++gj) {
      if (kFp8)
        wait_bar(cx, &bars.f8_full[gj % S], (gj / S) & 1, true);
      else
        wait_bar(cx, &bars.kv_full[gj % S], (gj / S) & 1, true);
    }
  }
  if (warp == 1 && lane == 0) {
    tc::commit(tc::smem_u32(&bars.drain));
    wait_bar(cx, &bars.drain, 0, true);
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

template <bool kFp8>
cudaError_t launch(const AttnParams& p, const CUtensorMap& tm_k,
                   const CUtensorMap& tm_v, cudaStream_t s) {
  using C = Cfg<kFp8>;
  // the shared-memory attribute was set on this device by ctas_per_sm(),
  // which sizing the grid always runs first (an attribute call per launch
  // costs microseconds of host time)
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg =
      pdl_config(dim3(p.grid), dim3(C::kThreads), C::kSmem, s, attr);
  return cudaLaunchKernelEx(&cfg, verify_split_tc_kernel<kFp8>, p, tm_k, tm_v);
}

template <bool kFp8>
int ctas_per_sm() {
  using C = Cfg<kFp8>;
  if (cudaFuncSetAttribute(verify_split_tc_kernel<kFp8>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::kSmem) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &n, verify_split_tc_kernel<kFp8>, C::kThreads, C::kSmem) !=
      cudaSuccess)
    return 0;
  return n < 1 ? 0 : 1;  // TMEM: one 512-column allocation per SM
}

}  // namespace

cudaError_t launch_verify_split_tc(const AttnParams& p, const CUtensorMap& tm_k,
                                   const CUtensorMap& tm_v, cudaStream_t s) {
  return p.k_scales ? launch<true>(p, tm_k, tm_v, s)
                    : launch<false>(p, tm_k, tm_v, s);
}

int verify_split_tc_ctas_per_sm(bool fp8) {
  return fp8 ? ctas_per_sm<true>() : ctas_per_sm<false>();
}

int verify_split_tc_box_rows(int page_size) { return page_size < kT ? page_size : kT; }

}  // namespace specv
