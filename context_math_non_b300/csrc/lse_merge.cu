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
// partial; the P loads of a group are issued back to back so they are in flight together.  The
// row's LSE values are read by all threads of the row (L1 broadcast).  Inputs are read once and
// output written once, so loads/stores use the streaming cache hints.

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

// VPR = 16-byte vectors per row (0 = runtime value `vpr`).
template <bool BF16, int VPR>
__global__ void __launch_bounds__(kMergeThreads)
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
    const float* lrow = lse_parts + r;
    float M = -INFINITY;
    for (int c = 0; c < P; ++c) M = fmaxf(M, __ldg(lrow + static_cast<long long>(c) * rows));
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    float W = 0.f;
    if (M != -INFINITY) {
      const float Ml2 = M * kLog2e;
      for (int c0 = 0; c0 < P; c0 += kGroup) {
        uint4 v[kGroup];
        float wgt[kGroup];
#pragma unroll
        for (int g = 0; g < kGroup; ++g) {
          if (c0 + g < P) {
            v[g] = __ldcs(o_parts + static_cast<long long>(c0 + g) * part_stride + i);
            wgt[g] = ptx::ex2(fmaf(__ldg(lrow + static_cast<long long>(c0 + g) * rows), kLog2e,
                                   -Ml2));
          }
        }
#pragma unroll
        for (int g = 0; g < kGroup; ++g) {
          if (c0 + g < P) {
            float f[8];
            unpack8<BF16>(v[g], f);
            W += wgt[g];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = fmaf(wgt[g], f[e], acc[e]);
          }
        }
      }
    }
    const float inv = M != -INFINITY ? 1.f / W : 0.f;
    uint4 out;
    out.x = ptx::pack2<BF16>(acc[0] * inv, acc[1] * inv);
    out.y = ptx::pack2<BF16>(acc[2] * inv, acc[3] * inv);
    out.z = ptx::pack2<BF16>(acc[4] * inv, acc[5] * inv);
    out.w = ptx::pack2<BF16>(acc[6] * inv, acc[7] * inv);
    __stcs(o + i, out);
    if (lse_out != nullptr && col == 0) lse_out[r] = M != -INFINITY ? M + logf(W) : -INFINITY;
  }
}

template <bool BF16, int VPR>
cudaError_t launch_merge_typed(const void* o_parts, const float* lse_parts, int P, long long rows,
                               int vpr, void* o, float* lse, cudaStream_t stream) {
  const long long total = rows * vpr;
  const int sms = device_sm_count();
  long long blocks = (total + kMergeThreads - 1) / kMergeThreads;
  const long long cap = static_cast<long long>(sms > 0 ? sms : 148) * 8;
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
