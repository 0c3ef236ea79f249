// Log-sum-exp merge of per-chunk partial attention outputs (HBM-bound streaming kernel).
//
// Ring Attention ("Scaling AI Inference Across Multiple GPUs Using NVIDIA TensorRT with
// Multi-Device Inference Support", subsection "Ring Attention") updates each query row's output
// as the K/V blocks of the other ranks stream past.  With the partial outputs O_c and their LSE_c
// available, the update is a weighted combination per row:
//   M = max_c LSE_c,  w_c = exp(LSE_c - M),  O = sum_c w_c O_c / sum_c w_c,
//   LSE = M + ln sum_c w_c.
//
// One thread owns one 16-byte vector (8 elements) of one row and streams that vector of every
// partial; the LSE values and O vectors of a group of partials are all issued before any is
// used, so they are in flight together.  The row's LSE values are read by all threads of the row
// (L1 broadcast).  Inputs are read once and output written once, so loads/stores use the
// streaming cache hints.

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "cpattn_internal.h"
#include "ptx_sm103.cuh"

namespace cpattn {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kGroup = 8;   // partial vectors loaded before any is consumed

template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (BF16) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    } else {
      __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      float2 x = __half22float2(h);
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
    }
  }
}

// VPR = 16-byte vectors per row (0 = runtime value `vpr`).  Partials are taken in groups of
// kGroup: all LSE values and O vectors of a group are loaded before any is used, and groups are
// combined with a running maximum (acc and W rescaled by exp(M_old - M_new) when it moves), which
// for P <= kGroup is exactly the one-pass formula.
template <bool BF16, int VPR>
__global__ void __launch_bounds__(kMergeThreads, 3)
    lse_merge_kernel(const uint4* __restrict__ o_parts, const float* __restrict__ lse_parts,
                     int P, long long rows, int vpr_rt, uint4* __restrict__ o,
                     float* __restrict__ lse_out) {
  const int vpr = VPR > 0 ? VPR : vpr_rt;
  const long long total = rows * vpr;
  const long long part_stride = total;  // uint4 elements per partial
  const float kLog2e = 1.4426950408889634f;
  for (long long i = static_cast<long long>(blockIdx.x) * kMergeThreads + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * kMergeThreads) {
    const long long r = i / vpr;
    const int col = static_cast<int>(i - r * vpr);
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    float W = 0.f;
    float Ml2 = -INFINITY;   // running max of LSE * log2(e)
    for (int c0 = 0; c0 < P; c0 += kGroup) {
      uint4 v[kGroup];
      float ls[kGroup];
#pragma unroll
      for (int g = 0; g < kGroup; ++g) {
        if (c0 + g < P) {
          ls[g] = __ldg(lse_parts + static_cast<long long>(c0 + g) * rows + r) * kLog2e;
          v[g] = __ldcs(o_parts + static_cast<long long>(c0 + g) * part_stride + i);
        } else {
          ls[g] = -INFINITY;
        }
      }
      float mg = ls[0];
#pragma unroll
      for (int g = 1; g < kGroup; ++g) mg = fmaxf(mg, ls[g]);
      const float m_new = fmaxf(Ml2, mg);
      if (m_new == -INFINITY) continue;        // every partial so far is empty
      if (m_new > Ml2) {
        const float sc = ptx::ex2(Ml2 - m_new);   // 0 while Ml2 = -inf
        W *= sc;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] *= sc;
        Ml2 = m_new;
      }
#pragma unroll
      for (int g = 0; g < kGroup; ++g) {
        if (c0 + g < P) {
          const float wgt = ptx::ex2(ls[g] - Ml2);
          float f[8];
          unpack8<BF16>(v[g], f);
          W += wgt;
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[e] = fmaf(wgt, f[e], acc[e]);
        }
      }
    }
    const bool empty = Ml2 == -INFINITY;
    const float inv = empty ? 0.f : 1.f / W;
    uint4 out;
    out.x = ptx::pack2<BF16>(acc[0] * inv, acc[1] * inv);
    out.y = ptx::pack2<BF16>(acc[2] * inv, acc[3] * inv);
    out.z = ptx::pack2<BF16>(acc[4] * inv, acc[5] * inv);
    out.w = ptx::pack2<BF16>(acc[6] * inv, acc[7] * inv);
    __stcs(o + i, out);
    if (lse_out != nullptr && col == 0)
      lse_out[r] = empty ? -INFINITY : (Ml2 + log2f(W)) * 0.69314718055994530942f;
  }
}

template <bool BF16, int VPR>
cudaError_t launch_merge_typed(const void* o_parts, const float* lse_parts, int P, long long rows,
                               int vpr, void* o, float* lse, cudaStream_t stream) {
  const long long total = rows * vpr;
  const int sms = device_sm_count();
  long long blocks = (total + kMergeThreads - 1) / kMergeThreads;
  const long long cap = static_cast<long long>(sms > 0 ? sms : 148) * 3;
  if (blocks > cap) blocks = cap;
  lse_merge_kernel<BF16, VPR><<<static_cast<int>(blocks), kMergeThreads, 0, stream>>>(
      static_cast<const uint4*>(o_parts), lse_parts, P, rows, vpr, static_cast<uint4*>(o), lse);
  return cudaGetLastError();
}

}  // namespace

attn_status launch_lse_merge(const void* o_parts, const float* lse_parts, int P, long long rows,
                             int D, bool bf16, void* o, float* lse, cudaStream_t stream) {
  const int vpr = D / 8;
  cudaError_t e;
  if (vpr == 16)
    e = bf16 ? launch_merge_typed<true, 16>(o_parts, lse_parts, P, rows, vpr, o, lse, stream)
             : launch_merge_typed<false, 16>(o_parts, lse_parts, P, rows, vpr, o, lse, stream);
  else if (vpr == 8)
    e = bf16 ? launch_merge_typed<true, 8>(o_parts, lse_parts, P, rows, vpr, o, lse, stream)
             : launch_merge_typed<false, 8>(o_parts, lse_parts, P, rows, vpr, o, lse, stream);
  else
    e = bf16 ? launch_merge_typed<true, 0>(o_parts, lse_parts, P, rows, vpr, o, lse, stream)
             : launch_merge_typed<false, 0>(o_parts, lse_parts, P, rows, vpr, o, lse, stream);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace cpattn
