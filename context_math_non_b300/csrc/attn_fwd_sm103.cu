// Non-causal attention forward on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Computes, for every query row, the attention over one contiguous KV range -- the whole
// sequence (P = 1) or one of P chunks, each chunk standing in for one step of Ring Attention
// ("Scaling AI Inference Across Multiple GPUs Using NVIDIA TensorRT with Multi-Device Inference
// Support", subsection "Ring Attention", Figure 3) -- with an online softmax, so the full score
// matrix never exists anywhere.  Outputs: O normalised over the range, and the range's
// natural-log LSE.  Variants of the same kernel (template parameters): the sequence-sharded
// (Ulysses) addressing (kSeq), the ring walk over all P chunks with the merge on chip (kRing),
// and e4m3 operands (kF8).
//
// Work unit: (chunk c, batch*head bh, 256-query block qb); in ring mode (bh, qb) over all chunks.
// A persistent grid of one CTA per SM walks the units in a static round-robin; consecutive units
// share (bh, c), so the CTAs resident at one time read the same K/V chunk and L2 serves the
// re-reads.
//
// CTA roles (384 threads = 3 warpgroups):
//   warps 0-3  softmax for query tile 0 (thread = row; TMEM lanes 0..127)
//   warps 4-7  softmax for query tile 1
//   warp  8    TMA producer: Q tiles once per unit, then K_j / V_j through a ring of stages
//   warp  9    TMEM allocation and MMA issue: the whole warp runs the loop (waits voted across
//              the warp) and one elected lane issues by predication, so the operands stay
//              warp-uniform
//   warp  10   with separate P (D = 64): issues the O += P V GEMMs while warp 9 issues S
//   warps 10-11 otherwise idle (they complete the third warpgroup, which releases registers to
//              the softmax warpgroups with setmaxnreg)
// Tensor memory (512 columns): S0 | S1 | O0 | O1.  For D = 128, P (16-bit, or e4m3) is written
// over the first part of its S columns and read from TMEM by the P*V MMA.  The MMA order per KV
// step j
//   O0 += P0 V_{j-1};  S0 = Q0 K_j^T;  O1 += P1 V_{j-1};  S1 = Q1 K_j^T
// lets each softmax warpgroup work on its tile while the tensor core runs the other tile's two
// GEMMs.  For D = 64 the O regions are half as wide and P gets its own columns, so S_t(j+1) is
// computed while the softmax of S_t(j) runs (separate-P schedule).  The running max is only moved
// (and O rescaled) when it grows by more than 2^8, so most steps skip the rescale; the final
// normalisation uses the same stale max, so results are exact.
//
// Shared memory: the two Q tiles, the K/V ring (4 stages of 32 KB at D = 128, 8 of 16 KB for
// D = 64 and e4m3) and, for 16-bit outputs in the plain layout, one 4 KB output staging region
// per softmax warp: a warp's 32 output rows leave through TMA stores instead of per-thread row
// stores (see the epilogue).
//
// Every wait is bounded (see mbar_wait): a lost signal ends the kernel with ATTN_ERR_TIMEOUT in
// the status word instead of a hang.

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <atomic>
#include <mutex>

#include "cpattn_internal.h"
#include "ptx_sm103.cuh"

namespace cpattn {

__device__ int g_attn_status = 0;

namespace {

constexpr int kBM = 128;          // query rows per tile (= TMEM lanes)
constexpr int kBN = 128;          // KV rows per tile
constexpr int kQT = 2;            // query tiles per CTA
constexpr int kHalfBytes = 128 * 128;  // [128 rows][64 x 16-bit] swizzled box = 16 KB
constexpr int kThreads = 384;
// Register split: the kernel is compiled for kLaunchRegs per thread (the 384-thread launch
// bound); the producer warpgroup gives registers back (setmaxnreg.dec) and the two softmax
// warpgroups take them (setmaxnreg.inc).  The increase must be covered by what is released,
// or setmaxnreg.inc would wait forever; the host refuses to launch a build whose register
// count differs from kLaunchRegs.
constexpr int kLaunchRegs = 168;
constexpr int kSoftmaxRegs = 192;
constexpr int kProducerRegs = 112;
static_assert(2 * 128 * (kSoftmaxRegs - kLaunchRegs) <= 128 * (kLaunchRegs - kProducerRegs),
              "setmaxnreg increase exceeds the registers released by the producer warpgroup");
static_assert(kLaunchRegs * kThreads <= 65536, "register file");

constexpr int kLoaderWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
// Schedules that run a unit's epilogue after the next unit's first tile (see the softmax loop).
constexpr bool kDeferEpilogueF8 = true;
constexpr bool kDeferEpilogue16 = false;
// Output rows are written with 32-byte stores when the output is 32-byte aligned.
constexpr bool kStore32 = true;
// 16-bit plain-layout kernels stage their output rows in shared memory and write them with TMA
// stores, 32 rows per warp (the e4m3 kernel measured slower with it and stores directly).
constexpr bool kStageStore = true;
constexpr int kStageWarpBytes = 32 * 128;   // 32 rows x one 64-column half of 16-bit O

// kF8: e4m3 operands (one byte per element), so a 128-row tile of D = 128 is one 128-byte-wide
// swizzled box of 16 KB, like a 16-bit tile of D = 64.
template <int D, bool kF8 = false>
struct Cfg {
  static constexpr int NH = kF8 ? 1 : D / 64;             // 128-byte-wide boxes per row
  static constexpr int TILE = NH * kHalfBytes;            // bytes of one 128-row tile
  static constexpr int STAGES = (TILE == kHalfBytes) ? 8 : 4;   // K/V ring depth
  static constexpr int NBARS = 2 * STAGES + 10 * kQT + 2;
  // output staging: one region per softmax warp (kStageStore)
  static constexpr bool STAGE_OUT = kStageStore && !kF8;
  static constexpr int OUT_STAGE = STAGE_OUT ? kQT * 4 * kStageWarpBytes : 0;
  static constexpr int SMEM = 1024 /*alignment slack*/ + kQT * TILE + STAGES * TILE +
                              OUT_STAGE + NBARS * 8 + 16;
  static constexpr uint32_t S_COL0 = 0, S_COL1 = 128, O_COL0 = 256, O_COL1 = 256 + D;
  // D = 64 leaves 128 columns free: P gets its own columns, so S(j+1) can be computed while the
  // softmax of S(j) runs (separate-P schedule).  D = 128 writes P over the first half of S.
  static constexpr bool SEP_P = (D == 64 && !kF8);
  static constexpr uint32_t P_COL0 = SEP_P ? 384 : S_COL0, P_COL1 = SEP_P ? 448 : S_COL1;
  static constexpr bool DEFER_EPILOGUE = kF8 ? kDeferEpilogueF8 : kDeferEpilogue16;
};

struct Params {
  int Sq, Skv, P, BH, n_qb;
  int num_units;     // BH * P * n_qb (< 2^31, checked on the host)
  int kv_q, kv_r;    // Skv = kv_q * P + kv_r
  float scale_log2;  // softmax scale * log2(e) (times the Q and K scales for e4m3 inputs)
  float o_scale;     // output multiplier: 1, or the V scale for e4m3 inputs
  int o_align32;     // o is 32-byte aligned: rows are written in whole 32-byte sectors
  void* o;           // [P][BH][Sq][D]  (sequence-sharded layout: see SeqLayout)
  float* lse;        // [P][BH][Sq] or null
  unsigned long long limit_ns;
  // Sequence-sharded (Ulysses) addressing, used by the kSeq kernels only: Q/K/V/O are
  // [R][B][S/R][H][D] for R ranks; attention head bh = (g*B + b)*(H/R) + j is head g*(H/R) + j
  // of batch b, and token t = r*(S/R) + s lives in rank r's shard.
  int sq_R, sq_B, sq_H, sq_Hl, sq_Sl, sq_box;
};

// Rows [row, row + 128) of head bh into one 64-column half of a swizzled tile.  The plain layout
// is one 3-D box; the sequence-sharded layout takes boxes of sq_box rows (never straddling two
// ranks' shards) from the 4-D map (D, H, S/R, R*B).  Rows past the end are zero-filled by TMA.
template <bool kSeq>
__device__ __forceinline__ void load_rows(uint8_t* dst, const CUtensorMap* map, int x, int row,
                                          int bh, uint64_t* bar, const Params& p) {
  if constexpr (!kSeq) {
    ptx::tma_load_3d(dst, map, x, row, bh, bar);
  } else {
    const int j = bh % p.sq_Hl;
    const int rb = bh / p.sq_Hl;
    const int b = rb % p.sq_B;
    const int g = rb / p.sq_B;
    const int h = g * p.sq_Hl + j;
    for (int r0 = 0; r0 < 128; r0 += p.sq_box) {
      const int t = row + r0;
      const int rank = t / p.sq_Sl;
      ptx::tma_load_4d(dst + r0 * 128, map, x, h, t - rank * p.sq_Sl, rank * p.sq_B + b, bar);
    }
  }
}

// Element offset of output row q_row of head bh (partial prow) in O.
template <bool kSeq, int D>
__device__ __forceinline__ long long out_row_offset(long long prow, int bh, int q_row,
                                                    const Params& p) {
  if constexpr (!kSeq) {
    return (prow * p.Sq + q_row) * static_cast<long long>(D);
  } else {
    const int j = bh % p.sq_Hl;
    const int rb = bh / p.sq_Hl;
    const int b = rb % p.sq_B;
    const int g = rb / p.sq_B;
    const int rank = q_row / p.sq_Sl;
    const long long tok = (static_cast<long long>(rank) * p.sq_B + b) * p.sq_Sl +
                          (q_row - rank * p.sq_Sl);
    return (tok * p.sq_H + g * p.sq_Hl + j) * static_cast<long long>(D);
  }
}

struct Unit {
  int qb, c, bh, lo, n, last_valid;
};

// Ring mode: the KV tiles of a unit, chunk by chunk in ring order.  Chunk c (the KV block rank c
// holds) is cut into 128-row tiles starting at its first row, the last tile masked at the chunk
// end; after the last tile of chunk c comes chunk c - 1 (mod P), as a rank receives its
// neighbour's block at each ring step.
struct KvCursor {
  int c, left, tile, nt, lo, last_valid;
};

// Chunk c covers KV rows [floor(c*Skv/P), floor((c+1)*Skv/P)); with Skv = q*P + r,
// floor(c*Skv/P) = c*q + floor(c*r/P), and c*r < P^2 <= 2^32 fits 32-bit unsigned arithmetic.
__device__ __forceinline__ int chunk_start(int c, const Params& p) {
  return c * p.kv_q + static_cast<int>((static_cast<uint32_t>(c) * static_cast<uint32_t>(p.kv_r)) /
                                       static_cast<uint32_t>(p.P));
}

__device__ __forceinline__ void cursor_load(KvCursor& k, const Params& p) {
  k.lo = chunk_start(k.c, p);
  const int len = chunk_start(k.c + 1, p) - k.lo;
  k.nt = (len + kBN - 1) / kBN;
  k.last_valid = len - (k.nt - 1) * kBN;
  k.tile = 0;
}
__device__ __forceinline__ void cursor_start(KvCursor& k, const Unit& w, const Params& p) {
  k.c = w.c;
  k.left = p.P;
  cursor_load(k, p);
}
__device__ __forceinline__ int cursor_row(const KvCursor& k) { return k.lo + k.tile * kBN; }
__device__ __forceinline__ int cursor_valid(const KvCursor& k) {
  return k.tile == k.nt - 1 ? k.last_valid : kBN;
}
__device__ __forceinline__ void cursor_next(KvCursor& k, const Params& p) {
  if (++k.tile == k.nt && --k.left > 0) {
    k.c = (k.c == 0 ? p.P : k.c) - 1;
    cursor_load(k, p);
  }
}

// Ring mode unit u = (bh, qb): all P chunks.  The block starts at the chunk of the rank that
// holds its first query row (queries split into P ranks like the keys), and the tile count is
// the sum over chunks: with Skv = q*P + r, r chunks have q + 1 rows and P - r have q.
__device__ __forceinline__ Unit decode_ring_unit(int u, const Params& p) {
  Unit w;
  const uint32_t uu = static_cast<uint32_t>(u);
  const uint32_t bh = uu / static_cast<uint32_t>(p.n_qb);
  w.qb = static_cast<int>(uu - bh * static_cast<uint32_t>(p.n_qb));
  w.bh = static_cast<int>(bh);
  const long long row0 = static_cast<long long>(w.qb) * (kQT * kBM);
  const long long c0 = ((row0 + 1) * p.P - 1) / p.Sq;
  w.c = static_cast<int>(c0 < p.P - 1 ? c0 : p.P - 1);
  w.lo = 0;
  w.n = (p.P - p.kv_r) * ((p.kv_q + kBN - 1) / kBN) + p.kv_r * ((p.kv_q + kBN) / kBN);
  w.last_valid = kBN;
  return w;
}

__device__ __forceinline__ Unit decode_unit(int u, const Params& p) {
  Unit w;
  const uint32_t uu = static_cast<uint32_t>(u);
  const uint32_t r = uu / static_cast<uint32_t>(p.n_qb);
  w.qb = static_cast<int>(uu - r * static_cast<uint32_t>(p.n_qb));
  const uint32_t bh = r / static_cast<uint32_t>(p.P);
  w.c = static_cast<int>(r - bh * static_cast<uint32_t>(p.P));
  w.bh = static_cast<int>(bh);
  w.lo = chunk_start(w.c, p);
  const int len = chunk_start(w.c + 1, p) - w.lo;
  w.n = (len + kBN - 1) / kBN;
  w.last_valid = len - (w.n - 1) * kBN;
  return w;
}

// Wait for an already-issued asynchronous completion regardless of the abort flag (used only to
// drain in-flight copies / MMAs before the CTA exits on the error path).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > limit_ns) return;
  }
}

template <int D>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[D]) {
  if constexpr (D == 128) {
    ptx::tmem_ld128(taddr, r);
  } else {
    ptx::tmem_ld64(taddr, r);
  }
}

// No-op hook for softmax_tile.
struct NoHook {
  __device__ __forceinline__ void operator()() const {}
};

// One KV tile of the online softmax for this thread's row: read the 128 logits from TMEM at
// s_addr (then run after_load: the logits are in registers; before_store runs before the first
// write to p_addr), update the running max m (only
// when it grows by more than the threshold; `need` reports a move and `alpha` = 2^(m_old -
// m_new), or 1), write P = 2^(s*scale*log2(e) - m) as 16-bit pairs to the 64 TMEM columns at
// p_addr, and return the row sum of P.  Columns >= valid count as -inf (last tile of a KV
// chunk); kMasked = false lets a caller that passes valid = 128 drop that branch at compile time.
template <bool BF16, bool kMasked, typename AfterLoad = NoHook, typename BeforeStore = NoHook,
          bool kP8 = false>
__device__ __forceinline__ float softmax_tile(uint32_t s_addr, uint32_t p_addr, float sl2,
                                              int valid, float& m, bool& need, float& alpha,
                                              AfterLoad after_load = AfterLoad(),
                                              BeforeStore before_store = BeforeStore()) {
  uint32_t sr[kBN];
  ptx::tmem_ld128(s_addr, sr);
  after_load();
  if (kMasked || valid < kBN) {
#pragma unroll
    for (int c = 0; c < kBN; ++c)
      if (c >= valid) sr[c] = __float_as_uint(-INFINITY);
  }
#define SV(c) __uint_as_float(sr[c])
  float mx0 = SV(0), mx1 = SV(1), mx2 = SV(2), mx3 = SV(3);
#pragma unroll
  for (int c = 4; c + 8 <= kBN; c += 8) {
    mx0 = ptx::max3(mx0, SV(c), SV(c + 1));
    mx1 = ptx::max3(mx1, SV(c + 2), SV(c + 3));
    mx2 = ptx::max3(mx2, SV(c + 4), SV(c + 5));
    mx3 = ptx::max3(mx3, SV(c + 6), SV(c + 7));
  }
  mx0 = ptx::max3(mx0, SV(kBN - 4), SV(kBN - 3));
  mx1 = ptx::max3(mx1, SV(kBN - 2), SV(kBN - 1));
  const float m_new = fmaxf(m, ptx::max3(mx0, mx1, fmaxf(mx2, mx3)) * sl2);
  need = m_new > m + kRescaleThreshold;
  alpha = need ? ptx::ex2(m - m_new) : 1.f;   // 0 on the first tile (m = -inf)
  if (need) m = m_new;
  // p = 2^(s*scale*log2(e) - m), two elements per packed fp32x2 FMA / ADD.
  const uint64_t sl2x2 = ptx::f2_pack(sl2, sl2);
  const uint64_t negm2 = ptx::f2_pack(-m, -m);
  uint64_t lacc[4];
#pragma unroll
  for (int a = 0; a < 4; ++a) lacc[a] = ptx::f2_pack(0.f, 0.f);
  if constexpr (kP8) {
    // P as e4m3, four per tensor-memory column (32 columns for the 128 keys)
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      uint32_t pk[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int e = 32 * h + 4 * c;
        const uint64_t xa = ptx::f2_fma(ptx::f2_pack(SV(e), SV(e + 1)), sl2x2, negm2);
        const uint64_t xb = ptx::f2_fma(ptx::f2_pack(SV(e + 2), SV(e + 3)), sl2x2, negm2);
        float x0, x1, x2, x3;
        ptx::f2_unpack(xa, x0, x1);
        ptx::f2_unpack(xb, x2, x3);
        const float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1), p2 = ptx::ex2(x2), p3 = ptx::ex2(x3);
        lacc[(2 * c) & 3] = ptx::f2_add(lacc[(2 * c) & 3], ptx::f2_pack(p0, p1));
        lacc[(2 * c + 1) & 3] = ptx::f2_add(lacc[(2 * c + 1) & 3], ptx::f2_pack(p2, p3));
        pk[c] = ptx::pack4_e4m3(p0, p1, p2, p3);
      }
      if (h == 0) before_store();
      ptx::tmem_st8(p_addr + 8 * h, pk);
    }
  } else {
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    uint32_t pk[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const int e = 32 * h + 2 * c;
      const uint64_t x = ptx::f2_fma(ptx::f2_pack(SV(e), SV(e + 1)), sl2x2, negm2);
      float x0, x1;
      ptx::f2_unpack(x, x0, x1);
      const float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
      lacc[c & 3] = ptx::f2_add(lacc[c & 3], ptx::f2_pack(p0, p1));
      pk[c] = ptx::pack2<BF16>(p0, p1);
    }
    if (h == 0) before_store();
    ptx::tmem_st16(p_addr + 16 * h, pk);
  }
  }
#undef SV
  float la, lb;
  ptx::f2_unpack(ptx::f2_add(ptx::f2_add(lacc[0], lacc[1]), ptx::f2_add(lacc[2], lacc[3])), la,
                 lb);
  return la + lb;
}

// O row *= alpha for this thread's TMEM lane, 64 columns per load round trip.
template <int D>
__device__ __forceinline__ void rescale_o(uint32_t o_addr, float alpha) {
  const uint64_t a2 = ptx::f2_pack(alpha, alpha);
#pragma unroll
  for (int half = 0; half < D / 64; ++half) {
    uint32_t r[64];
    ptx::tmem_ld64(o_addr + 64 * half, r);
#pragma unroll
    for (int c = 0; c < 64; c += 2) {
      float x0, x1;
      ptx::f2_unpack(
          ptx::f2_mul(ptx::f2_pack(__uint_as_float(r[c]), __uint_as_float(r[c + 1])), a2), x0,
          x1);
      r[c] = __float_as_uint(x0);
      r[c + 1] = __float_as_uint(x1);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t q[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) q[c] = r[16 * i + c];
      ptx::tmem_st16(o_addr + 64 * half + 16 * i, q);
    }
  }
}

template <int D, bool BF16, bool kSeq, bool kRing, bool kF8 = false>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_o, const Params p) {
  using C = Cfg<D, kF8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + kQT * C::TILE;
  uint8_t* sOut = sKV + C::STAGES * C::TILE;   // 1024-byte aligned (tiles are 16 KB multiples)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sOut + C::OUT_STAGE);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = bars + C::STAGES;
  uint64_t* q_full = bars + 2 * C::STAGES;
  uint64_t* q_empty = q_full + kQT;
  uint64_t* s_full = q_empty + kQT;
  uint64_t* p_full = s_full + kQT;
  uint64_t* o_full = p_full + kQT;
  uint64_t* o_empty = o_full + kQT;
  uint64_t* s_free = o_empty + kQT;     // separate-P schedule: S tile read into registers
  uint64_t* pv_done = s_free + kQT;     // separate-P schedule: P*V of the tile completed
  uint64_t* mma_drain = pv_done + kQT;   // [0]: MMA warp, [1]: P*V warp (separate-P schedule)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t lim = p.limit_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(&kv_full[s], 1);
      ptx::mbar_init(&kv_empty[s], 1);
    }
    for (int t = 0; t < kQT; ++t) {
      ptx::mbar_init(&q_full[t], 1);
      ptx::mbar_init(&q_empty[t], 1);
      ptx::mbar_init(&s_full[t], 1);
      ptx::mbar_init(&p_full[t], 4);
      ptx::mbar_init(&o_full[t], 1);
      ptx::mbar_init(&o_empty[t], 4);
      ptx::mbar_init(&s_free[t], 4);
      ptx::mbar_init(&pv_done[t], 1);
    }
    ptx::mbar_init(&mma_drain[0], 1);
    ptx::mbar_init(&mma_drain[1], 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(tmem_slot, kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == kLoaderWarp && lane == 0) {
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_v);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 8) {
    // Producer warpgroup: hand registers to the softmax warpgroups.
    ptx::regs_dec<kProducerRegs>();
  if (warp == kLoaderWarp) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t kv_pos = 0, it = 0;
      int q_issued[kQT];
      for (int t = 0; t < kQT; ++t) q_issued[t] = -1;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x, ++it) {
        const Unit w = kRing ? decode_ring_unit(u, p) : decode_unit(u, p);
        for (int t = 0; ok && t < kQT; ++t) {
          ok = ptx::mbar_wait(&q_empty[t], (it & 1) ^ 1, abort_flag, &g_attn_status, lim);
          if (!ok) break;
          q_issued[t] = static_cast<int>(it);
          ptx::mbar_arrive_expect_tx(&q_full[t], C::TILE);
          for (int h = 0; h < C::NH; ++h)
            load_rows<kSeq>(sQ + t * C::TILE + h * kHalfBytes, &tm_q, 64 * h,
                            w.qb * (kQT * kBM) + t * kBM, w.bh, &q_full[t], p);
        }
        KvCursor kc;
        if constexpr (kRing) cursor_start(kc, w, p);
        for (int j = 0; ok && j < w.n; ++j) {
          const int kv_row = kRing ? cursor_row(kc) : w.lo + j * kBN;
          if constexpr (kRing) cursor_next(kc, p);
          for (int which = 0; which < 2; ++which) {
            const uint32_t st = kv_pos % C::STAGES;
            const uint32_t ph = (kv_pos / C::STAGES) & 1;
            ok = ptx::mbar_wait(&kv_empty[st], ph ^ 1, abort_flag, &g_attn_status, lim);
            if (!ok) break;
            ptx::mbar_arrive_expect_tx(&kv_full[st], C::TILE);
            const CUtensorMap* map = which == 0 ? &tm_k : &tm_v;
            if (kF8 && which == 1) {
              // V^T [BH][D][Skv]: the box is 128 keys (x, a multiple of 16 bytes) x D rows
              ptx::tma_load_3d(sKV + st * C::TILE, map, kv_row, 0, w.bh, &kv_full[st]);
            } else {
              for (int h = 0; h < C::NH; ++h)
                load_rows<kSeq>(sKV + st * C::TILE + h * kHalfBytes, map, 64 * h, kv_row, w.bh,
                                &kv_full[st], p);
            }
            ++kv_pos;
          }
        }
      }
      if (!ok) {
        // Error path: let every copy this thread issued land before the CTA's memory goes away.
        const uint32_t issued = kv_pos < static_cast<uint32_t>(C::STAGES) ? kv_pos : C::STAGES;
        for (uint32_t i = kv_pos - issued; i < kv_pos; ++i)
          drain_wait(&kv_full[i % C::STAGES], (i / C::STAGES) & 1, lim);
        for (int t = 0; t < kQT; ++t)
          if (q_issued[t] >= 0) drain_wait(&q_full[t], q_issued[t] & 1, lim);
      }
    }
  } else if (warp == kMmaWarp || (C::SEP_P && warp == kMmaWarp + 1)) {
    // ------------------------------------------------------------------ MMA issuers
    // The whole warp runs its loop with identical control flow (every wait is voted across
    // the warp); one lane issues every MMA and commit.  With separate P the S = Q K^T
    // GEMMs (this warp) and the O += P V GEMMs (the next warp) touch disjoint tensor-memory
    // columns and are ordered only through the softmax hand-offs, so two warps issue them:
    // each issuing warp is a serial chain of waits and issues, and splitting it halves the
    // chain per KV step.
    {
      // The issuing lane, chosen once (the warp stays converged through the whole loop), or an
      // elect.sync per instruction: chosen per schedule and GEMM by measurement.  With one
      // issuing warp the single elect is ≈ 3-4 % faster; with the two warps of separate P it
      // gains ≈ 1 % for the S GEMMs and loses for the P*V GEMMs and the commits.
      constexpr bool kElectOnce = !C::SEP_P;   // for the P*V GEMMs and the commits
      const uint32_t lead = ptx::elect_leader();
      auto mma_ss = [&](uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
        ptx::mma_ss_lead(lead, d, a, b, id, acc);
      };
      auto mma_ts = [&](uint32_t d, uint32_t a, uint64_t b, uint32_t id, uint32_t acc) {
        if constexpr (kElectOnce) ptx::mma_ts_lead(lead, d, a, b, id, acc);
        else ptx::mma_ts_elect(d, a, b, id, acc);
      };
      auto commit = [&](uint64_t* bar) {
        if constexpr (kElectOnce) ptx::mma_commit_lead(lead, bar);
        else ptx::mma_commit_elect(bar);
      };
      // e4m3 (kF8): format code 0 in both operand fields and a K-major B (V^T) for P*V
      constexpr uint32_t kIdescS = ptx::idesc_f16(kF8 ? false : BF16, false, kBM, kBN);
      constexpr uint32_t kIdescPV = ptx::idesc_f16(kF8 ? false : BF16, !kF8, kBM, D);
      const uint32_t sQ_addr = ptx::smem_u32(sQ);
      const uint32_t sKV_addr = ptx::smem_u32(sKV);

      auto issue_s = [&](int t, uint32_t st) {
        const uint32_t a0 = sQ_addr + t * C::TILE;
        const uint32_t b0 = sKV_addr + st * C::TILE;
        const uint32_t d_s = tmem + (t == 0 ? C::S_COL0 : C::S_COL1);
        const uint64_t da = ptx::smem_desc_sw128(a0, 16, 1024);
        const uint64_t db = ptx::smem_desc_sw128(b0, 16, 1024);
        if constexpr (kF8) {
          // K = 32 one-byte elements per MMA: four 32-byte steps inside the 128-byte rows, one
          // assembly block (measured +2.5 % over one MMA per block for this schedule)
          static_assert(D == 128 && !C::SEP_P, "e4m3 path: D = 128, one issuing warp");
          ptx::gemm_ss_f8_d128(lead, d_s, da, db, kIdescS);
        } else {
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            // descriptor start-address field counts 16-byte units; no carry can leave it
            const uint64_t off =
                static_cast<uint64_t>(((ks >> 2) * kHalfBytes + (ks & 3) * 32) >> 4);
            mma_ss(d_s, da + off, db + off, kIdescS, ks > 0);
          }
        }
      };
      auto issue_pv = [&](int t, uint32_t st, bool acc) {
        const uint32_t b0 = sKV_addr + st * C::TILE;
        const uint32_t d_o = tmem + (t == 0 ? C::O_COL0 : C::O_COL1);
        const uint32_t a_p = tmem + (t == 0 ? C::P_COL0 : C::P_COL1);
        if constexpr (kF8) {
          // A = P (e4m3, 8 columns per 32 keys), B = the V^T tile, K-major over the keys
          const uint64_t dvt = ptx::smem_desc_sw128(b0, 16, 1024);
          ptx::gemm_ts_f8_n128(lead, d_o, a_p, dvt, kIdescPV, acc ? 1u : 0u);
        } else {
          const uint64_t dv = ptx::smem_desc_sw128(b0, kHalfBytes, 1024);
#pragma unroll
          for (int ks = 0; ks < kBN / 16; ++ks) {
            mma_ts(d_o, a_p + ks * 8, dv + static_cast<uint64_t>(ks * 128), kIdescPV,
                              (acc || ks > 0) ? 1u : 0u);
          }
        }
      };

      uint32_t kv_pos = 0, it = 0, pph[2] = {0, 0};
      bool ok = true;
      auto wait_kv = [&](uint32_t& st) -> bool {
        st = kv_pos % C::STAGES;
        const uint32_t ph = (kv_pos / C::STAGES) & 1;
        ++kv_pos;
        return __all_sync(0xffffffffu,
                          ptx::mbar_wait(&kv_full[st], ph, abort_flag, &g_attn_status, lim));
      };

      uint32_t sfph[2] = {0, 0};
      auto vote_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu,
                          ptx::mbar_wait(bar, parity, abort_flag, &g_attn_status, lim));
      };
      if constexpr (C::SEP_P) {
        // The loader fills ring positions K_0, V_0, K_1, V_1, ...; with an even number of
        // stages the K tiles always land in even stages (consumed here by the S warp) and the
        // V tiles in odd ones (the P*V warp), so each stage has one consumer.
        static_assert(C::STAGES % 2 == 0, "K and V stages must alternate");
        const bool s_role = warp == kMmaWarp;
        uint32_t pos = s_role ? 0u : 1u;   // ring position of this warp's next tile
        auto wait_tile = [&](uint32_t& st) -> bool {
          st = pos % C::STAGES;
          const uint32_t ph = (pos / C::STAGES) & 1;
          pos += 2;
          return vote_wait(&kv_full[st], ph);
        };
        for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x, ++it) {
          const Unit w = kRing ? decode_ring_unit(u, p) : decode_unit(u, p);
          for (int j = 0; ok && j < w.n; ++j) {
            uint32_t st;
            if (!(ok = wait_tile(st))) break;
            for (int t = 0; t < kQT; ++t) {
              if (s_role) {
                // S_t(j) overwrites the S columns of S_t(j-1) (or of the previous unit's last
                // tile): wait until the softmax has them in registers.
                if (j > 0 || it > 0) {
                  if (!(ok = vote_wait(&s_free[t], sfph[t]))) break;
                  sfph[t] ^= 1;
                }
                if (j == 0 && !(ok = vote_wait(&q_full[t], it & 1))) break;
                ptx::tc_fence_after();
                issue_s(t, st);
                commit(&s_full[t]);
                if (j == w.n - 1) commit(&q_empty[t]);
              } else {
                if (!(ok = vote_wait(&p_full[t], pph[t]))) break;
                pph[t] ^= 1;
                if (j == 0 && it > 0 && !(ok = vote_wait(&o_empty[t], (it - 1) & 1))) break;
                ptx::tc_fence_after();
                issue_pv(t, st, j > 0);
                commit(&pv_done[t]);
                if (j == w.n - 1) commit(&o_full[t]);
              }
            }
            if (!ok) break;
            commit(&kv_empty[st]);
          }
        }
        // All MMAs this warp issued complete before TMEM is released.
        commit(&mma_drain[s_role ? 0 : 1]);
        drain_wait(&mma_drain[s_role ? 0 : 1], 0, lim);
      } else {
      for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x, ++it) {
        const Unit w = kRing ? decode_ring_unit(u, p) : decode_unit(u, p);
        uint32_t sk, sv;
        if (!(ok = wait_kv(sk))) break;
        for (int t = 0; t < kQT; ++t) {
          if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(&q_full[t], it & 1, abort_flag,
                                                             &g_attn_status, lim))))
            break;
          ptx::tc_fence_after();
          issue_s(t, sk);
          commit(&s_full[t]);
          if (w.n == 1) commit(&q_empty[t]);
        }
        if (!ok) break;
        commit(&kv_empty[sk]);

        for (int j = 1; ok && j <= w.n; ++j) {
          if (!(ok = wait_kv(sv))) break;
          for (int t = 0; t < kQT; ++t) {
            if (!(ok = __all_sync(0xffffffffu, ptx::mbar_wait(&p_full[t], pph[t], abort_flag,
                                                               &g_attn_status, lim))))
              break;
            pph[t] ^= 1;
            if (j == 1 && it > 0) {
              if (!(ok = __all_sync(0xffffffffu,
                                    ptx::mbar_wait(&o_empty[t], (it - 1) & 1, abort_flag,
                                                   &g_attn_status, lim))))
                break;
            }
            ptx::tc_fence_after();
            issue_pv(t, sv, j > 1);
            if (t == kQT - 1) commit(&kv_empty[sv]);
            if (j == w.n) {
              commit(&o_full[t]);
            } else {
              if (t == 0 && !(ok = wait_kv(sk))) break;
              issue_s(t, sk);
              commit(&s_full[t]);
              if (j == w.n - 1) commit(&q_empty[t]);
              if (t == kQT - 1) commit(&kv_empty[sk]);
            }
          }
        }
      }
      // All MMAs this warp issued complete before TMEM is released.
      commit(&mma_drain[0]);
      drain_wait(&mma_drain[0], 0, lim);
      }
    }
  }
  } else {
    // ------------------------------------------------------------------ softmax warpgroups
    ptx::regs_inc<kSoftmaxRegs>();
    const int t = warp >> 2;                    // query tile of this warpgroup
    const int wq = warp & 3;                    // TMEM lane quarter
    const int row = wq * 32 + lane;             // row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + (t == 0 ? C::S_COL0 : C::S_COL1);
    const uint32_t o_addr = tmem + lane_base + (t == 0 ? C::O_COL0 : C::O_COL1);
    const uint32_t p_addr = tmem + lane_base + (t == 0 ? C::P_COL0 : C::P_COL1);
    const float sl2 = p.scale_log2;
    uint32_t sph = 0, oph = 0, it = 0, pdph = 0;
    bool ok = true;
    bool pv_pending = false;   // separate-P schedule: a P*V of this tile may still read P

    // Separate-P schedule hooks (no-ops when P overwrites S): release the S columns as soon as
    // the logits are in registers; before overwriting P, wait for the P*V that reads it.
    auto after_load = [&]() {
      if constexpr (C::SEP_P) {
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&s_free[t]);
      }
    };
    auto before_store = [&]() {
      if constexpr (C::SEP_P) {
        if (pv_pending) {
          ok = __all_sync(0xffffffffu,
                          ptx::mbar_wait(&pv_done[t], pdph, abort_flag, &g_attn_status, lim));
          pdph ^= 1;
          ptx::tc_fence_after();
        }
        pv_pending = true;
      }
    };

    // ---------------------------------------------------------------- epilogue
    // Output of unit w: normalised O row and LSE.  With DEFER_EPILOGUE it runs after the next
    // unit's first tile has been handed to the MMA warp, so the wait for the unit's last P*V
    // and the stores overlap the next unit's GEMMs instead of delaying its first softmax (a
    // unit's first tile never touches O: it is only overwritten by that tile's P*V, which waits
    // for o_empty).
    auto epilogue = [&](const Unit& w, float m, float l) {
      ok = __all_sync(0xffffffffu,
                      ptx::mbar_wait(&o_full[t], oph, abort_flag, &g_attn_status, lim));
      if (!ok) return;
      oph ^= 1;
      ptx::tc_fence_after();
      const int q_row = w.qb * (kQT * kBM) + t * kBM + row;
      const bool valid = q_row < p.Sq;
      const float inv_l = p.o_scale / l;
      const long long prow = static_cast<long long>(kRing ? 0 : w.c) * p.BH + w.bh;
      uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) +
                       out_row_offset<kSeq, D>(prow, w.bh, valid ? q_row : 0, p);
      // The whole O row goes to registers first, so the accumulator is released (o_empty)
      // before the normalisation and the global stores: the next output's first P*V, which
      // overwrites O, waits only for the tensor-memory reads.
      uint32_t orr[D];
      tmem_ld_cols<D>(o_addr, orr);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&o_empty[t]);
      if constexpr (C::STAGE_OUT && !kSeq) {
        // The warp's 32 rows go through its shared-memory region, one 64-column half at a time
        // (128-byte swizzled rows: conflict-free 16-byte writes), and leave as one TMA store per
        // half: whole, coalesced lines; rows past Sq are clipped by the tensor map.
        uint8_t* stg = sOut + warp * kStageWarpBytes;
        const uint32_t stg_row = ptx::smem_u32(stg) + lane * 128;
        const int row0 = w.qb * (kQT * kBM) + t * kBM + wq * 32;
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          if (lane == 0) ptx::bulk_wait_read_all();   // the region's previous store has read it
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t pk[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
              pk[i] = ptx::pack2<BF16>(__uint_as_float(orr[64 * h + 8 * c + 2 * i]) * inv_l,
                                       __uint_as_float(orr[64 * h + 8 * c + 2 * i + 1]) * inv_l);
            ptx::st_shared_v4(stg_row + ((c ^ (lane & 7)) << 4), pk[0], pk[1], pk[2], pk[3]);
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && row0 < p.Sq) {   // a box that starts inside the tensor
            ptx::tma_store_3d(&tm_o, stg, 64 * h, row0, static_cast<int>(prow));
            ptx::bulk_commit();
          }
        }
      } else if (valid && p.o_align32) {
        // 32-byte stores: each writes a whole sector of the row (a thread owns one row)
#pragma unroll
        for (int v = 0; v < D / 16; ++v) {
          uint32_t pk[8];
#pragma unroll
          for (int c = 0; c < 8; ++c)
            pk[c] = ptx::pack2<BF16>(__uint_as_float(orr[16 * v + 2 * c]) * inv_l,
                                     __uint_as_float(orr[16 * v + 2 * c + 1]) * inv_l);
          ptx::st_global_v8(orow + 16 * v, pk);
        }
      } else if (valid) {
        uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
        for (int v = 0; v < D / 8; ++v) {
          uint32_t pk[4];
#pragma unroll
          for (int c = 0; c < 4; ++c)
            pk[c] = ptx::pack2<BF16>(__uint_as_float(orr[8 * v + 2 * c]) * inv_l,
                                     __uint_as_float(orr[8 * v + 2 * c + 1]) * inv_l);
          dst[v] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
      if (valid && p.lse != nullptr)
        p.lse[prow * p.Sq + q_row] = (m + __log2f(l)) * 0.69314718055994530942f;
    };
    bool pending = false;   // DEFER_EPILOGUE: the previous unit's epilogue has not run yet
    Unit w_prev{};
    float m_prev = 0.f, l_prev = 1.f;

    for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x, ++it) {
      const Unit w = kRing ? decode_ring_unit(u, p) : decode_unit(u, p);
      float m = -INFINITY;   // running max of scaled logits, log2 units
      float l = 0.f;         // running denominator relative to m
      KvCursor kc;
      if constexpr (kRing) cursor_start(kc, w, p);
      for (int j = 0; j < w.n; ++j) {
        ok = __all_sync(0xffffffffu,
                        ptx::mbar_wait(&s_full[t], sph, abort_flag, &g_attn_status, lim));
        if (!ok) break;
        sph ^= 1;
        ptx::tc_fence_after();

        bool need;
        float alpha;
        int valid;
        if constexpr (kRing) {
          valid = cursor_valid(kc);
          cursor_next(kc, p);
        } else {
          valid = j == w.n - 1 ? w.last_valid : kBN;
        }
        // One instantiation with a run-time mask branch keeps the kernel's code small enough
        // for the instruction cache with one issuing warp (≈ +4 % at D = 128); the two-warp
        // separate-P schedule measures faster with a masked and an unmasked instantiation.
        float l_tile;
        if constexpr (C::SEP_P) {
          l_tile = valid < kBN
                       ? softmax_tile<BF16, true, decltype(after_load), decltype(before_store),
                                      kF8>(s_addr, p_addr, sl2, valid, m, need, alpha,
                                           after_load, before_store)
                       : softmax_tile<BF16, false, decltype(after_load), decltype(before_store),
                                      kF8>(s_addr, p_addr, sl2, kBN, m, need, alpha, after_load,
                                           before_store);
        } else {
          l_tile = softmax_tile<BF16, false, decltype(after_load), decltype(before_store), kF8>(
              s_addr, p_addr, sl2, valid, m, need, alpha, after_load, before_store);
        }
        if (!ok) break;
        l = l * alpha + l_tile;
        // Rescale O when the max moved in any row of this warp.  O is not in use: the P*V of
        // earlier steps completed before S_j was signalled (P over S), or before pv_done was
        // observed above (separate P); this step's P*V is only issued after the arrive below.
        if (j > 0 && __any_sync(0xffffffffu, need)) rescale_o<D>(o_addr, alpha);
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&p_full[t]);
        if (C::DEFER_EPILOGUE && j == 0 && pending) {
          pending = false;
          epilogue(w_prev, m_prev, l_prev);
          if (!ok) break;
        }
      }
      if (!ok) break;
      if constexpr (C::DEFER_EPILOGUE) {
        pending = true;
        w_prev = w;
        m_prev = m;
        l_prev = l;
      } else {
        epilogue(w, m, l);
      }
    }
    if (C::DEFER_EPILOGUE && ok && pending) epilogue(w_prev, m_prev, l_prev);
    // this warp's output stores finish before the CTA (and its shared memory) goes away
    if (C::STAGE_OUT && !kSeq && lane == 0) ptx::bulk_wait_all();
  }


  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}



// ----------------------------------------------------------------------------- CTA-pair kernel
// D = 128 variant that runs the tensor core in CTA pairs (cta_group::2, a cluster of two CTAs):
// each MMA is M = 256 -- 128 query rows from each CTA -- and the B operand (a K tile for
// S = Q K^T, a V tile for O += P V) is split along N between the two CTAs.  So each CTA loads
// only half of every K/V tile (K: 64 of the 128 KV rows; V: 64 of the 128 columns of D) and
// reads only its half from shared memory for the MMA: shared-memory traffic for B operands and
// TMA writes per SM are halved (TMA writes competing with the MMA operand reads cost the
// single-CTA kernel 5-10 %).  The cross-SM hand-offs cost more than that saves, so this variant
// is slower and not the default (attn_set_kernel_variant).
//
// Unit: (chunk, batch*head, 512-query block); CTA r of the pair owns query rows
// [256 r, 256 r + 256) of the block as two 128-row tiles, exactly like the single-CTA kernel.
// Roles per CTA as in the single-CTA kernel, plus warp 10 = relay: the even ("leader") CTA's
// MMA thread issues for both CTAs, so it must know that both CTAs' operands have landed; each
// CTA's relay thread waits for its own TMA completions and arrives on the leader's barriers.
// Softmax warps of both CTAs publish P and release O on the leader's barriers (remote arrive
// for the odd CTA); the leader's commits are multicast to the barriers of both CTAs.
constexpr int kPairStages = 10;
constexpr int kPairStageBytes = 16 * 1024;   // K half [64 rows][128 d] or V half [128 rows][64 d]
constexpr int kPairQBytes = 128 * 128 * 2;   // one 128-row Q tile, D = 128
constexpr int kRelayWarp = 10;
constexpr int kPairNBars = 3 * kPairStages + 9 * kQT + 1;
constexpr int kPairSmem =
    1024 + kQT * kPairQBytes + kPairStages * kPairStageBytes + kPairNBars * 8 + 16;
static_assert(kPairSmem <= 232448, "shared memory per CTA");

template <bool BF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    attn_fwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const Params p) {
  constexpr int D = 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + kQT * kPairQBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sKV + kPairStages * kPairStageBytes);
  uint64_t* kv_full = bars;                        // local TMA completion
  uint64_t* kv_empty = kv_full + kPairStages;      // leader commit (multicast)
  uint64_t* kv_ready = kv_empty + kPairStages;     // leader only: both halves landed
  uint64_t* q_full = kv_ready + kPairStages;
  uint64_t* q_empty = q_full + kQT;
  uint64_t* q_ready = q_empty + kQT;               // leader only
  uint64_t* s_full = q_ready + kQT;
  uint64_t* p_full = s_full + kQT;                 // leader only, 8 arrivals
  uint64_t* o_full = p_full + kQT;
  uint64_t* o_empty = o_full + kQT;                // leader only, 8 arrivals
  uint64_t* mma_drain = o_empty + kQT;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kPairNBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t lim = p.limit_ns;
  const uint32_t rank = ptx::cluster_ctarank();
  const int cluster_id = static_cast<int>(blockIdx.x >> 1);
  const int n_clusters = static_cast<int>(gridDim.x >> 1);
  auto leader_addr = [&](const uint64_t* bar) { return ptx::mapa(ptx::smem_u32(bar), 0); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      ptx::mbar_init(&kv_full[s], 1);
      ptx::mbar_init(&kv_empty[s], 1);
      ptx::mbar_init(&kv_ready[s], 2);
    }
    for (int t = 0; t < kQT; ++t) {
      ptx::mbar_init(&q_full[t], 1);
      ptx::mbar_init(&q_empty[t], 1);
      ptx::mbar_init(&q_ready[t], 2);
      ptx::mbar_init(&s_full[t], 1);
      ptx::mbar_init(&p_full[t], 8);
      ptx::mbar_init(&o_full[t], 1);
      ptx::mbar_init(&o_empty[t], 8);
    }
    ptx::mbar_init(mma_drain, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc_pair(tmem_slot, kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  if (warp == kLoaderWarp && lane == 0) {
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_v);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();   // both CTAs' barriers exist before any remote arrive
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 8) {
    ptx::regs_dec<kProducerRegs>();
    if (warp == kLoaderWarp && lane == 0) {
      // ---------------------------------------------------------------- TMA producer (both)
      uint32_t st = 0, ph = 0, it = 0, issued_total = 0;
      int q_issued[kQT] = {-1, -1};
      bool ok = true;
      auto next_stage = [&](uint32_t& s_out, uint32_t& ph_out) -> bool {
        s_out = st;
        ph_out = ph;
        if (++st == kPairStages) {
          st = 0;
          ph ^= 1;
        }
        return ptx::mbar_wait<true>(&kv_empty[s_out], ph_out ^ 1, abort_flag, &g_attn_status, lim);
      };
      for (int u = cluster_id; ok && u < p.num_units; u += n_clusters, ++it) {
        const Unit w = decode_unit(u, p);
        for (int t = 0; ok && t < kQT; ++t) {
          ok = ptx::mbar_wait<true>(&q_empty[t], (it & 1) ^ 1, abort_flag, &g_attn_status, lim);
          if (!ok) break;
          q_issued[t] = static_cast<int>(it);
          ptx::mbar_arrive_expect_tx(&q_full[t], kPairQBytes);
          const int row = w.qb * (4 * kBM) + static_cast<int>(rank) * (kQT * kBM) + t * kBM;
          for (int h = 0; h < 2; ++h)
            ptx::tma_load_3d(sQ + t * kPairQBytes + h * kHalfBytes, &tm_q, 64 * h, row, w.bh,
                             &q_full[t]);
        }
        for (int j = 0; ok && j < w.n; ++j) {
          uint32_t s, sph;
          // K: this CTA's 64 of the tile's 128 KV rows, both 64-column halves of D
          if (!(ok = next_stage(s, sph))) break;
          ptx::mbar_arrive_expect_tx(&kv_full[s], kPairStageBytes);
          const int krow = w.lo + j * kBN + static_cast<int>(rank) * 64;
          for (int h = 0; h < 2; ++h)
            ptx::tma_load_3d(sKV + s * kPairStageBytes + h * (kPairStageBytes / 2), &tm_k, 64 * h,
                             krow, w.bh, &kv_full[s]);
          ++issued_total;
          // V: all 128 KV rows, this CTA's 64 columns of D
          if (!(ok = next_stage(s, sph))) break;
          ptx::mbar_arrive_expect_tx(&kv_full[s], kPairStageBytes);
          ptx::tma_load_3d(sKV + s * kPairStageBytes, &tm_v, 64 * static_cast<int>(rank),
                           w.lo + j * kBN, w.bh, &kv_full[s]);
          ++issued_total;
        }
      }
      if (!ok) {
        const uint32_t n = issued_total < kPairStages ? issued_total : kPairStages;
        for (uint32_t i = issued_total - n; i < issued_total; ++i)
          drain_wait(&kv_full[i % kPairStages], (i / kPairStages) & 1, lim);
        for (int t = 0; t < kQT; ++t)
          if (q_issued[t] >= 0) drain_wait(&q_full[t], q_issued[t] & 1, lim);
      }
    } else if (warp == kRelayWarp && lane == 0) {
      // ---------------------------------------------------------------- relay (both CTAs)
      uint32_t st = 0, ph = 0, it = 0;
      bool ok = true;
      for (int u = cluster_id; ok && u < p.num_units; u += n_clusters, ++it) {
        const Unit w = decode_unit(u, p);
        for (int t = 0; ok && t < kQT; ++t) {
          ok = ptx::mbar_wait<true>(&q_full[t], it & 1, abort_flag, &g_attn_status, lim);
          if (ok) ptx::mbar_arrive_cluster(leader_addr(&q_ready[t]));
        }
        for (int j = 0; ok && j < 2 * w.n; ++j) {
          ok = ptx::mbar_wait<true>(&kv_full[st], ph, abort_flag, &g_attn_status, lim);
          if (!ok) break;
          ptx::mbar_arrive_cluster(leader_addr(&kv_ready[st]));
          if (++st == kPairStages) {
            st = 0;
            ph ^= 1;
          }
        }
      }
    } else if (warp == kMmaWarp && lane == 0 && rank == 0) {
      // ---------------------------------------------------------------- MMA issuer (leader)
      constexpr uint32_t kIdescS = ptx::idesc_f16(BF16, false, 2 * kBM, kBN);
      constexpr uint32_t kIdescPV = ptx::idesc_f16(BF16, true, 2 * kBM, D);
      const uint32_t sQ_addr = ptx::smem_u32(sQ);
      const uint32_t sKV_addr = ptx::smem_u32(sKV);
      const uint32_t s_col[2] = {Cfg<D>::S_COL0, Cfg<D>::S_COL1};
      const uint32_t o_col[2] = {Cfg<D>::O_COL0, Cfg<D>::O_COL1};
      constexpr uint16_t kBoth = 0x3;

      auto issue_s = [&](int t, uint32_t stg) {
        const uint32_t a0 = sQ_addr + t * kPairQBytes;
        const uint32_t b0 = sKV_addr + stg * kPairStageBytes;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          ptx::mma_ss_pair(
              tmem + s_col[t],
              ptx::smem_desc_sw128(a0 + (ks >> 2) * kHalfBytes + (ks & 3) * 32, 16, 1024),
              ptx::smem_desc_sw128(b0 + (ks >> 2) * (kPairStageBytes / 2) + (ks & 3) * 32, 16,
                                   1024),
              kIdescS, ks > 0);
        }
      };
      auto issue_pv = [&](int t, uint32_t stg, bool acc) {
        const uint32_t b0 = sKV_addr + stg * kPairStageBytes;
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks) {
          ptx::mma_ts_pair(tmem + o_col[t], tmem + s_col[t] + ks * 8,
                           ptx::smem_desc_sw128(b0 + ks * 2048, kHalfBytes, 1024), kIdescPV,
                           (acc || ks > 0) ? 1u : 0u);
        }
      };

      uint32_t kst = 0, kph = 0, it = 0, pph[2] = {0, 0};
      bool ok = true;
      auto wait_kv = [&](uint32_t& stg) -> bool {
        stg = kst;
        const uint32_t ph = kph;
        if (++kst == kPairStages) {
          kst = 0;
          kph ^= 1;
        }
        return ptx::mbar_wait<true>(&kv_ready[stg], ph, abort_flag, &g_attn_status, lim);
      };

      for (int u = cluster_id; ok && u < p.num_units; u += n_clusters, ++it) {
        const Unit w = decode_unit(u, p);
        uint32_t sk, sv;
        if (!(ok = wait_kv(sk))) break;
        for (int t = 0; t < kQT; ++t) {
          if (!(ok = ptx::mbar_wait<true>(&q_ready[t], it & 1, abort_flag, &g_attn_status, lim))) break;
          ptx::tc_fence_after();
          issue_s(t, sk);
          ptx::mma_commit_pair(&s_full[t], kBoth);
          if (w.n == 1) ptx::mma_commit_pair(&q_empty[t], kBoth);
        }
        if (!ok) break;
        ptx::mma_commit_pair(&kv_empty[sk], kBoth);

        for (int j = 1; ok && j <= w.n; ++j) {
          if (!(ok = wait_kv(sv))) break;
          for (int t = 0; t < kQT; ++t) {
            if (!(ok = ptx::mbar_wait<true>(&p_full[t], pph[t], abort_flag, &g_attn_status, lim)))
              break;
            pph[t] ^= 1;
            if (j == 1 && it > 0) {
              if (!(ok = ptx::mbar_wait<true>(&o_empty[t], (it - 1) & 1, abort_flag, &g_attn_status,
                                        lim)))
                break;
            }
            ptx::tc_fence_after();
            issue_pv(t, sv, j > 1);
            if (t == kQT - 1) ptx::mma_commit_pair(&kv_empty[sv], kBoth);
            if (j == w.n) {
              ptx::mma_commit_pair(&o_full[t], kBoth);
            } else {
              if (t == 0 && !(ok = wait_kv(sk))) break;
              issue_s(t, sk);
              ptx::mma_commit_pair(&s_full[t], kBoth);
              if (j == w.n - 1) ptx::mma_commit_pair(&q_empty[t], kBoth);
              if (t == kQT - 1) ptx::mma_commit_pair(&kv_empty[sk], kBoth);
            }
          }
        }
      }
      ptx::mma_commit_pair(mma_drain, 0x1);
      drain_wait(mma_drain, 0, lim);
    }
  } else {
    // ------------------------------------------------------------------ softmax (both CTAs)
    ptx::regs_inc<kSoftmaxRegs>();
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + (t == 0 ? Cfg<D>::S_COL0 : Cfg<D>::S_COL1);
    const uint32_t o_addr = tmem + lane_base + (t == 0 ? Cfg<D>::O_COL0 : Cfg<D>::O_COL1);
    const uint32_t p_full_leader = leader_addr(&p_full[t]);
    const uint32_t o_empty_leader = leader_addr(&o_empty[t]);
    const float sl2 = p.scale_log2;
    uint32_t sph = 0, oph = 0;
    bool ok = true;

    for (int u = cluster_id; ok && u < p.num_units; u += n_clusters) {
      const Unit w = decode_unit(u, p);
      float m = -INFINITY;
      float l = 0.f;
      for (int j = 0; j < w.n; ++j) {
        ok = __all_sync(0xffffffffu,
                        ptx::mbar_wait<true>(&s_full[t], sph, abort_flag, &g_attn_status, lim));
        if (!ok) break;
        sph ^= 1;
        ptx::tc_fence_after();
        bool need;
        float alpha;
        const float l_tile =
            (j == w.n - 1 && w.last_valid < kBN)
                ? softmax_tile<BF16, true>(s_addr, s_addr, sl2, w.last_valid, m, need, alpha)
                : softmax_tile<BF16, false>(s_addr, s_addr, sl2, kBN, m, need, alpha);
        l = l * alpha + l_tile;
        if (j > 0 && __any_sync(0xffffffffu, need)) rescale_o<D>(o_addr, alpha);
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_cluster(p_full_leader);
      }
      if (!ok) break;

      ok = __all_sync(0xffffffffu,
                      ptx::mbar_wait<true>(&o_full[t], oph, abort_flag, &g_attn_status, lim));
      if (!ok) break;
      oph ^= 1;
      ptx::tc_fence_after();
      const int q_row = w.qb * (4 * kBM) + static_cast<int>(rank) * (kQT * kBM) + t * kBM + row;
      const bool valid = q_row < p.Sq;
      const float inv_l = 1.f / l;
      const long long prow = static_cast<long long>(w.c) * p.BH + w.bh;
      uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) +
                       (prow * p.Sq + (valid ? q_row : 0)) * static_cast<long long>(D);
#pragma unroll
      for (int half = 0; half < D / 64; ++half) {
        uint32_t orr[64];
        ptx::tmem_ld64(o_addr + 64 * half, orr);
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + 64 * half);
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            uint32_t pk[4];
#pragma unroll
            for (int c = 0; c < 4; ++c)
              pk[c] = ptx::pack2<BF16>(__uint_as_float(orr[8 * v + 2 * c]) * inv_l,
                                       __uint_as_float(orr[8 * v + 2 * c + 1]) * inv_l);
            dst[v] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        }
      }
      if (valid && p.lse != nullptr)
        p.lse[prow * p.Sq + q_row] = (m + __log2f(l)) * 0.69314718055994530942f;
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(o_empty_leader);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();   // the leader's MMAs on this CTA's memory are complete
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// Watchdog self-test: one thread waits on a barrier nobody arrives on.
__global__ void watchdog_selftest_kernel(unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    (void)ptx::mbar_wait(&bar, 0, &abort_flag, &g_attn_status, limit_ns);
  }
}

// --------------------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 3-D map over a [BH][S][D] 16-bit tensor, box = 64 elements x box_rows rows x 1, 128-byte
// swizzle.
bool make_map(CUtensorMap* map, const void* base, bool bf16, int D, int S, int BH,
              int box_rows = 128) {
  auto enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                           static_cast<cuuint64_t>(S) * static_cast<cuuint64_t>(D) * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                   3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// One-time set-up of a kernel on the current device: the dynamic shared-memory limit above 48 KB
// is a per-device attribute, so it is set once for every device the process launches on, and the
// kernel's register count is checked against the register split.  Thread-safe.
constexpr int kMaxDevices = 64;
struct KernelSetup {
  std::once_flag once[kMaxDevices];
  cudaError_t err[kMaxDevices] = {};
};

template <typename Kernel>
cudaError_t setup_kernel(KernelSetup& s, Kernel kern, int smem_bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::call_once(s.once[dev], [&] {
    cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem_bytes);
    cudaFuncAttributes fa;
    if (r == cudaSuccess) r = cudaFuncGetAttributes(&fa, kern);
    // see the register split: setmaxnreg needs exactly the launch register count
    if (r == cudaSuccess && fa.numRegs != kLaunchRegs) r = cudaErrorInvalidKernelImage;
    s.err[dev] = r;
  });
  return s.err[dev];
}

template <bool BF16>
cudaError_t launch_pair(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                        const Params& p, int grid, cudaStream_t stream) {
  auto kern = attn_fwd_pair_kernel<BF16>;
  static KernelSetup setup;
  const cudaError_t e = setup_kernel(setup, kern, kPairSmem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, kPairSmem, stream>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

// mo: the output as [rows][Sq][D] 16-bit, box 64 columns x 32 rows (the staged TMA stores of the
// plain layout; not read by the sequence-sharded kernels).
template <int D, bool BF16, bool kSeq = false, bool kRing = false, bool kF8 = false>
cudaError_t launch_typed(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                         const CUtensorMap& mo, const Params& p, int grid, cudaStream_t stream) {
  auto kern = attn_fwd_kernel<D, BF16, kSeq, kRing, kF8>;
  static KernelSetup setup;
  const cudaError_t e = setup_kernel(setup, kern, Cfg<D, kF8>::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, Cfg<D, kF8>::SMEM, stream>>>(mq, mk, mv, mo, p);
  return cudaGetLastError();
}

}  // namespace

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

namespace {
std::atomic<int> g_variant{0};
}  // namespace

int set_attention_variant(int v) { return g_variant.exchange(v); }

attn_status launch_attention(const void* q, const void* k, const void* v, void* o, float* lse,
                             int P, int B, int H, int Sq, int Skv, int D, bool bf16, float scale,
                             cudaStream_t stream, unsigned long long limit_ns, int max_ctas,
                             bool ring) {
  const int BH = B * H;
  int sms = device_sm_count();
  if (sms <= 0) return ATTN_ERR_CUDA;
  if (max_ctas > 0 && max_ctas < sms) sms = max_ctas;
  // D = 128 runs on CTA pairs (needs at least one pair of SMs); D = 64 on single CTAs.
  const bool pair = !ring && D == 128 && g_variant.load() == 1 && sms >= 2;
  const int rows_per_unit = pair ? 4 * kBM : kQT * kBM;
  CUtensorMap mq, mk, mv, mo;
  if (!make_map(&mq, q, bf16, D, Sq, BH) || !make_map(&mk, k, bf16, D, Skv, BH, pair ? 64 : 128) ||
      !make_map(&mv, v, bf16, D, Skv, BH) ||
      !make_map(&mo, o, bf16, D, Sq, ring ? BH : P * BH, 32))
    return ATTN_ERR_CUDA;
  Params p;
  p.Sq = Sq;
  p.Skv = Skv;
  p.P = P;
  p.BH = BH;
  p.n_qb = (Sq + rows_per_unit - 1) / rows_per_unit;
  const long long units = static_cast<long long>(BH) * (ring ? 1 : P) * p.n_qb;
  if (units >= (1ll << 31) || P > 65536) return ATTN_ERR_UNSUPPORTED;
  p.num_units = static_cast<int>(units);
  p.kv_q = Skv / P;
  p.kv_r = Skv % P;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.o_scale = 1.f;
  p.o = o;
  p.o_align32 = (reinterpret_cast<uintptr_t>(o) & 31u) == 0 && kStore32 ? 1 : 0;
  p.lse = lse;
  p.limit_ns = limit_ns;
  cudaError_t e;
  if (pair) {
    const int pairs = p.num_units < sms / 2 ? p.num_units : sms / 2;
    e = bf16 ? launch_pair<true>(mq, mk, mv, p, 2 * pairs, stream)
             : launch_pair<false>(mq, mk, mv, p, 2 * pairs, stream);
  } else {
    const int grid = p.num_units < sms ? p.num_units : sms;
    if (ring) {
      if (D == 128)
        e = bf16 ? launch_typed<128, true, false, true>(mq, mk, mv, mo, p, grid, stream)
                 : launch_typed<128, false, false, true>(mq, mk, mv, mo, p, grid, stream);
      else
        e = bf16 ? launch_typed<64, true, false, true>(mq, mk, mv, mo, p, grid, stream)
                 : launch_typed<64, false, false, true>(mq, mk, mv, mo, p, grid, stream);
    } else if (D == 128) {
      e = bf16 ? launch_typed<128, true>(mq, mk, mv, mo, p, grid, stream)
               : launch_typed<128, false>(mq, mk, mv, mo, p, grid, stream);
    } else {
      e = bf16 ? launch_typed<64, true>(mq, mk, mv, mo, p, grid, stream)
               : launch_typed<64, false>(mq, mk, mv, mo, p, grid, stream);
    }
  }
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

namespace {
// 4-D map over a sequence-sharded [R][B][S/R][H][D] 16-bit tensor as (D, H, S/R, R*B), box =
// 64 elements x 1 head x box_rows tokens x 1, 128-byte swizzle.
bool make_seq_map(CUtensorMap* map, const void* base, bool bf16, int D, int H, int Sl, int RB,
                  int box_rows) {
  auto enc = get_encode_fn();
  if (!enc) return false;
  const cuuint64_t e = 2;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(Sl), static_cast<cuuint64_t>(RB)};
  cuuint64_t strides[3] = {D * e, static_cast<cuuint64_t>(H) * D * e,
                           static_cast<cuuint64_t>(Sl) * H * D * e};
  cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
             const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

attn_status launch_attention_ulysses(const void* q, const void* k, const void* v, void* o,
                                     float* lse, int R, int B, int S, int H, int D, bool bf16,
                                     float scale, cudaStream_t stream,
                                     unsigned long long limit_ns, int max_ctas) {
  const int Sl = S / R, Hl = H / R;
  int box = 128;
  while (box >= 16 && Sl % box != 0) box >>= 1;
  if (box < 16) return ATTN_ERR_UNSUPPORTED;
  CUtensorMap mq, mk, mv;
  if (!make_seq_map(&mq, q, bf16, D, H, Sl, R * B, box) ||
      !make_seq_map(&mk, k, bf16, D, H, Sl, R * B, box) ||
      !make_seq_map(&mv, v, bf16, D, H, Sl, R * B, box))
    return ATTN_ERR_CUDA;
  const CUtensorMap& mo = mq;   // the sequence-sharded kernels store O directly
  int sms = device_sm_count();
  if (sms <= 0) return ATTN_ERR_CUDA;
  if (max_ctas > 0 && max_ctas < sms) sms = max_ctas;
  Params p;
  p.Sq = S;
  p.Skv = S;
  p.P = 1;
  p.BH = B * H;                      // R*B*(H/R) attention heads
  p.n_qb = (S + kQT * kBM - 1) / (kQT * kBM);
  const long long units = static_cast<long long>(p.BH) * p.n_qb;
  if (units >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
  p.num_units = static_cast<int>(units);
  p.kv_q = S;
  p.kv_r = 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.o_scale = 1.f;
  p.o = o;
  p.o_align32 = (reinterpret_cast<uintptr_t>(o) & 31u) == 0 && kStore32 ? 1 : 0;
  p.lse = lse;
  p.limit_ns = limit_ns;
  p.sq_R = R;
  p.sq_B = B;
  p.sq_H = H;
  p.sq_Hl = Hl;
  p.sq_Sl = Sl;
  p.sq_box = box;
  const int grid = p.num_units < sms ? p.num_units : sms;
  cudaError_t e;
  if (D == 128)
    e = bf16 ? launch_typed<128, true, true>(mq, mk, mv, mo, p, grid, stream)
             : launch_typed<128, false, true>(mq, mk, mv, mo, p, grid, stream);
  else
    e = bf16 ? launch_typed<64, true, true>(mq, mk, mv, mo, p, grid, stream)
             : launch_typed<64, false, true>(mq, mk, mv, mo, p, grid, stream);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

namespace {
// 3-D map over a one-byte tensor [BH][rows][cols] (cols contiguous, a multiple of 16), box =
// 128 columns x 128 rows x 1, 128-byte swizzle.
bool make_map_u8(CUtensorMap* map, const void* base, int cols, int rows, int BH) {
  auto enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols),
                           static_cast<cuuint64_t>(rows) * static_cast<cuuint64_t>(cols)};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

attn_status launch_attention_fp8(const void* q, const void* k, const void* vt, void* o,
                                 float* lse, int P, int B, int H, int Sq, int Skv, float scale,
                                 float q_scale, float k_scale, float v_scale, cudaStream_t stream,
                                 unsigned long long limit_ns, int max_ctas) {
  constexpr int D = 128;
  const int BH = B * H;
  int sms = device_sm_count();
  if (sms <= 0) return ATTN_ERR_CUDA;
  if (max_ctas > 0 && max_ctas < sms) sms = max_ctas;
  CUtensorMap mq, mk, mv, mo;
  if (!make_map_u8(&mq, q, D, Sq, BH) || !make_map_u8(&mk, k, D, Skv, BH) ||
      !make_map_u8(&mv, vt, Skv, D, BH) || !make_map(&mo, o, true, D, Sq, BH, 32))
    return ATTN_ERR_CUDA;
  Params p;
  p.Sq = Sq;
  p.Skv = Skv;
  p.P = P;
  p.BH = BH;
  p.n_qb = (Sq + kQT * kBM - 1) / (kQT * kBM);
  const long long units = static_cast<long long>(BH) * p.n_qb;
  if (units >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
  p.num_units = static_cast<int>(units);
  p.kv_q = Skv / P;
  p.kv_r = Skv % P;
  p.scale_log2 = scale * q_scale * k_scale * 1.4426950408889634f;
  p.o_scale = v_scale;
  p.o = o;
  p.o_align32 = (reinterpret_cast<uintptr_t>(o) & 31u) == 0 && kStore32 ? 1 : 0;
  p.lse = lse;
  p.limit_ns = limit_ns;
  const int grid = p.num_units < sms ? p.num_units : sms;
  const cudaError_t e = launch_typed<D, true, false, true, true>(mq, mk, mv, mo, p, grid, stream);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status launch_watchdog_selftest(unsigned long long limit_ns, cudaStream_t stream) {
  watchdog_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status read_and_clear_device_status(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_CUDA;
  int h = 0;
  if (cudaMemcpyFromSymbol(&h, g_attn_status, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
  if (h != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_attn_status, &zero, sizeof(int)) != cudaSuccess)
      return ATTN_ERR_CUDA;
  }
  return static_cast<attn_status>(h);
}

}  // namespace cpattn
