// DeepSpeed Ulysses re-partition as an on-device layout permutation (HBM-bound copy kernel).
//
// "Scaling AI Inference Across Multiple GPUs Using NVIDIA TensorRT with Multi-Device Inference
// Support", subsection "DeepSpeed Ulysses" and Figure 4: an all-to-all before attention turns
// sequence sharding into head sharding, and a second one after attention turns it back.  With all
// P ranks' shards in one device buffer the all-to-all is a pure index permutation:
//   seq-sharded  X[p][b][s][h][d]  (rank p holds tokens p*S/P + s, all H heads)
//   head-sharded Y[g][b][j][t][d]  (rank g holds heads g*H/P + j, all S tokens)
//   Y[g][b][j][p*S/P + s][d] = X[p][b][s][g*H/P + j][d].
//
// Rows of a power-of-two number of 16-byte vectors (every D here) go through a tiled kernel whose
// blocks each own one (rank, head) pair and a run of tokens, so the index arithmetic is a few
// multiply-adds per vector.  Other row sizes use a general kernel whose threads walk one side's
// index space linearly; the matching vector on the other side is part of a run of D*elem_bytes
// contiguous bytes, so both sides are accessed in whole 16-byte vectors and in runs of at least
// one (token, head) row.

#include <cuda_runtime.h>

#include <cstdint>

#include "cpattn_internal.h"

namespace cpattn {
namespace {

constexpr int kLayoutThreads = 256;
constexpr int kUnroll = 4;
constexpr bool kSeq2HeadWalksHead = true;   // seq2head walks its destination (head-sharded) space
// Tiled kernel: adjacent heads a block moves together (their rows are contiguous in the
// sequence-sharded layout); the largest power of two up to this that divides H/P is used.
constexpr int kLayoutHeads = 4;

// kHeadLinear: threads walk the head-sharded index space linearly (true) or the sequence-sharded
// one (false); the other side is then accessed in runs of one (token, head) row.
template <typename Idx, bool kSeq2Head, bool kHeadLinear>
__global__ void __launch_bounds__(kLayoutThreads)
    layout_kernel(const uint4* __restrict__ in, uint4* __restrict__ out, Idx total, int B, int Hl,
                  int S, int Sl, int H, int vpr) {
  const Idx step = static_cast<Idx>(gridDim.x) * kLayoutThreads;
  for (Idx base = static_cast<Idx>(blockIdx.x) * kLayoutThreads * kUnroll + threadIdx.x;
       base < total; base += step * kUnroll) {
    uint4 v[kUnroll];
    Idx dst[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const Idx i = base + static_cast<Idx>(u) * kLayoutThreads;
      if (i < total) {
        Idx head_i, seq_i;
        if constexpr (kHeadLinear) {
          // head-sharded coordinates of vector i: [g][b][j][t][x]
          Idx r = i / vpr;
          const Idx x = i - r * vpr;
          const Idx t = r % S;
          r /= S;
          const Idx j = r % Hl;
          r /= Hl;
          const Idx b = r % B;
          const Idx g = r / B;
          const Idx p = t / Sl;
          const Idx s = t - p * Sl;
          head_i = i;
          seq_i = ((((p * B + b) * Sl + s) * H) + g * Hl + j) * vpr + x;
        } else {
          // sequence-sharded coordinates of vector i: [p][b][s][h][x]
          Idx r = i / vpr;
          const Idx x = i - r * vpr;
          const Idx h = r % H;
          r /= H;
          const Idx s = r % Sl;
          r /= Sl;
          const Idx b = r % B;
          const Idx p = r / B;
          const Idx g = h / Hl;
          const Idx j = h - g * Hl;
          seq_i = i;
          head_i = (((g * B + b) * Hl + j) * S + p * Sl + s) * vpr + x;
        }
        if constexpr (kSeq2Head) {
          v[u] = __ldcs(in + seq_i);
          dst[u] = head_i;
        } else {
          v[u] = __ldcs(in + head_i);
          dst[u] = seq_i;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const Idx i = base + static_cast<Idx>(u) * kLayoutThreads;
      if (i < total) __stcs(out + dst[u], v[u]);
    }
  }
}

// Tiled form for rows of a power-of-two number of vectors (vpr = 2^vpr_log2 <= 256): block
// (p, sb) x (g, b, j) moves tokens s in [sb*TT, (sb+1)*TT) of rank p for head j of rank g, batch b,
// TT = kUnroll * 256 / vpr.  All coordinates come from the block index, so a vector costs a few
// multiply-adds instead of the general kernel's chain of divisions; the head-sharded side of a
// block is one contiguous run of TT rows, the sequence-sharded side TT rows H*vpr vectors apart.
template <bool kSeq2Head>
__global__ void __launch_bounds__(kLayoutThreads)
    layout_tile_kernel(const uint4* __restrict__ in, uint4* __restrict__ out, int B, int Hl, int S,
                       int Sl, int H, int vpr_log2, int hb_log2, int nsb) {
  // block: rank p, token run sb, and heads j0 .. j0 + 2^hb_log2 - 1 of rank g, batch b
  const int Hg = Hl >> hb_log2;                 // head groups per (rank, batch)
  const int gbjg = blockIdx.y;                  // (g * B + b) * Hg + jg
  const int jg = gbjg % Hg;
  const int gb = gbjg / Hg;
  const int b = gb % B;
  const int g = gb / B;
  const int j0 = jg << hb_log2;
  const int p = blockIdx.x / nsb;
  const int sb = blockIdx.x - p * nsb;
  const int c_log2 = vpr_log2 + hb_log2;        // vectors of one token over the block's heads
  const int rows = kLayoutThreads >> c_log2;    // token rows per pass of the block
  const int c = threadIdx.x & ((1 << c_log2) - 1);
  const int rl = threadIdx.x >> c_log2;
  const int jj = c >> vpr_log2;                 // head of the group this thread moves
  const int x = c & ((1 << vpr_log2) - 1);
  // row indices of token s = 0 on both sides: the sequence-sharded side starts at the group's
  // first head (the group's rows are contiguous there), the head-sharded side at this head
  const long long seq_row0 = static_cast<long long>(p * B + b) * Sl * H + g * Hl + j0;
  const long long head_row0 = static_cast<long long>(gb * Hl + j0 + jj) * S +
                              static_cast<long long>(p) * Sl;
  uint4 v[kUnroll];
  long long dst[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int s = (sb * kUnroll + u) * rows + rl;
    if (s < Sl) {
      const long long seq_i = ((seq_row0 + static_cast<long long>(s) * H) << vpr_log2) + c;
      const long long head_i = ((head_row0 + s) << vpr_log2) + x;
      v[u] = __ldcs(in + (kSeq2Head ? seq_i : head_i));
      dst[u] = kSeq2Head ? head_i : seq_i;
    }
  }
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int s = (sb * kUnroll + u) * rows + rl;
    if (s < Sl) __stcs(out + dst[u], v[u]);
  }
}

template <typename Idx>
cudaError_t launch_layout_typed(const void* in, void* out, long long total, int B, int Hl, int S,
                                int Sl, int H, int vpr, bool seq2head, cudaStream_t stream) {
  const int sms = device_sm_count();
  long long blocks = (total + kLayoutThreads * kUnroll - 1) / (kLayoutThreads * kUnroll);
  const long long cap = static_cast<long long>(sms > 0 ? sms : 148) * 16;
  if (blocks > cap) blocks = cap;
  // Both directions write linearly (the destination is walked in order) and gather the source
  // in runs of one (token, head) row.
  if (seq2head)
    layout_kernel<Idx, true, kSeq2HeadWalksHead><<<static_cast<int>(blocks), kLayoutThreads, 0,
                                                   stream>>>(
        static_cast<const uint4*>(in), static_cast<uint4*>(out), static_cast<Idx>(total), B, Hl,
        S, Sl, H, vpr);
  else
    layout_kernel<Idx, false, !kSeq2HeadWalksHead><<<static_cast<int>(blocks), kLayoutThreads, 0,
                                                     stream>>>(
        static_cast<const uint4*>(in), static_cast<uint4*>(out), static_cast<Idx>(total), B, Hl,
        S, Sl, H, vpr);
  return cudaGetLastError();
}

}  // namespace

attn_status launch_layout(const void* in, void* out, int P, int B, int S, int H, int D,
                          int elem_bytes, bool seq2head, cudaStream_t stream) {
  const int vpr = D * elem_bytes / 16;
  const int Hl = H / P;
  const int Sl = S / P;
  const long long total = static_cast<long long>(P) * B * Hl * S * vpr;
  cudaError_t e;
  int vpr_log2 = 0;
  while ((1 << vpr_log2) < vpr) ++vpr_log2;
  int hb_log2 = 0;
  while ((2 << hb_log2) <= kLayoutHeads && Hl % (2 << hb_log2) == 0 &&
         (vpr << (hb_log2 + 1)) <= kLayoutThreads)
    ++hb_log2;
  const long long heads = (static_cast<long long>(P) * B * Hl) >> hb_log2;   // head groups
  if ((1 << vpr_log2) == vpr && vpr <= kLayoutThreads && heads <= 65535) {
    const int tokens_per_block = kUnroll * (kLayoutThreads / (vpr << hb_log2));
    const int nsb = (Sl + tokens_per_block - 1) / tokens_per_block;
    const dim3 grid(static_cast<unsigned>(static_cast<long long>(P) * nsb),
                    static_cast<unsigned>(heads));
    if (seq2head)
      layout_tile_kernel<true><<<grid, kLayoutThreads, 0, stream>>>(
          static_cast<const uint4*>(in), static_cast<uint4*>(out), B, Hl, S, Sl, H, vpr_log2, hb_log2,
          nsb);
    else
      layout_tile_kernel<false><<<grid, kLayoutThreads, 0, stream>>>(
          static_cast<const uint4*>(in), static_cast<uint4*>(out), B, Hl, S, Sl, H, vpr_log2, hb_log2,
          nsb);
    e = cudaGetLastError();
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
  }
  // 32-bit index arithmetic when every index (all bounded by total) and the loop counter, which
  // can step past total by one grid stride, stay far below 2^32.
  if (total < (1ll << 31))
    e = launch_layout_typed<uint32_t>(in, out, total, B, Hl, S, Sl, H, vpr, seq2head, stream);
  else
    e = launch_layout_typed<unsigned long long>(in, out, total, B, Hl, S, Sl, H, vpr, seq2head,
                                                stream);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace cpattn
