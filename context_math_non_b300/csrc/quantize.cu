// Per-tensor e4m3 quantization for the FP8 attention path: the absolute maximum of a 16-bit
// tensor (from which the caller picks the scale, e.g. amax / 448), and the conversion
// y = e4m3(x * inv_scale) -- fp32 multiply, round to nearest even, saturate to +-448 -- either in
// place order ([BH][S][D] -> [BH][S][D], for Q and K) or transposed per head ([BH][S][D] ->
// [BH][D][S], for V: the P*V GEMM takes V as a K-major operand over the keys).
// All three are HBM-bound streaming kernels.

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "cpattn_internal.h"
#include "ptx_sm103.cuh"

namespace cpattn {
namespace {

template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (BF16) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    } else {
      const __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      const float2 t = __half22float2(h);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
}

// Grid-stride max of |x| over n16 16-byte vectors; one atomic per block on the bit pattern of
// a non-negative float (ordered like the value).
template <bool BF16>
__global__ void __launch_bounds__(256) absmax_kernel(const uint4* __restrict__ in, long long n16,
                                                     unsigned int* out) {
  float m = 0.f;
  for (long long i = blockIdx.x * 256ll + threadIdx.x; i < n16; i += gridDim.x * 256ll) {
    float f[8];
    unpack8<BF16>(__ldg(in + i), f);
#pragma unroll
    for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(f[k]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float wm[8];
  if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = wm[0];
    for (int w = 1; w < 8; ++w) b = fmaxf(b, wm[w]);
    atomicMax(out, __float_as_uint(b));
  }
}

// Same order: each thread converts 16 elements (two 16-byte loads, one 16-byte store).
template <bool BF16>
__global__ void __launch_bounds__(256) quantize_kernel(const uint4* __restrict__ in,
                                                       uint4* __restrict__ out, long long n16x2,
                                                       float inv_scale) {
  for (long long i = blockIdx.x * 256ll + threadIdx.x; i < n16x2; i += gridDim.x * 256ll) {
    float a[8], b[8];
    unpack8<BF16>(__ldg(in + 2 * i), a);
    unpack8<BF16>(__ldg(in + 2 * i + 1), b);
    uint4 r;
    r.x = ptx::pack4_e4m3(a[0] * inv_scale, a[1] * inv_scale, a[2] * inv_scale, a[3] * inv_scale);
    r.y = ptx::pack4_e4m3(a[4] * inv_scale, a[5] * inv_scale, a[6] * inv_scale, a[7] * inv_scale);
    r.z = ptx::pack4_e4m3(b[0] * inv_scale, b[1] * inv_scale, b[2] * inv_scale, b[3] * inv_scale);
    r.w = ptx::pack4_e4m3(b[4] * inv_scale, b[5] * inv_scale, b[6] * inv_scale, b[7] * inv_scale);
    out[i] = r;
  }
}

// Transposed per head: block = one 128 (tokens) x 64 (features) tile of one head.  Thread
// (tq, fo) loads 4 tokens x 8 features (four 16-byte vectors; the 8 threads of a token row
// cover its 128 bytes) and packs, per feature, its 4 tokens' e4m3 bytes into one 32-bit word.
// Shared memory holds [64 features][128 tokens] bytes with the 16-byte chunks of feature row r
// XOR-swizzled by r / 8, so the word stores (one chunk per feature octet) and the 16-byte
// loads of the read-out are both free of bank conflicts; each output row of 128 tokens is then
// written as eight 16-byte vectors.
constexpr int kTT = 128, kTF = 64;
template <bool BF16>
__global__ void __launch_bounds__(256) quantize_t_kernel(const uint16_t* __restrict__ in,
                                                         uint8_t* __restrict__ out, int BH, int S,
                                                         int D, float inv_scale) {
  __shared__ __align__(16) uint32_t tile[kTF * kTT / 4];   // [feature][32 words of 4 tokens]
  const int s0 = blockIdx.x * kTT, d0 = blockIdx.y * kTF;
  const int tq = threadIdx.x >> 3, fo = threadIdx.x & 7;     // token quad, feature octet
  for (long long head = blockIdx.z; head < BH; head += gridDim.z) {
    const uint16_t* src = in + head * S * static_cast<long long>(D);
    uint8_t* dst = out + head * D * static_cast<long long>(S);
    __syncthreads();   // the previous head's tile has been read out
    float f[4][8];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int s = s0 + 4 * tq + r;
      if (s < S) {
        unpack8<BF16>(__ldg(reinterpret_cast<const uint4*>(src + static_cast<long long>(s) * D +
                                                          d0 + 8 * fo)),
                      f[r]);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) f[r][k] = 0.f;
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int row = 8 * fo + k;                       // feature within the tile
      const int word = tq;                              // tokens 4 tq .. 4 tq + 3
      const int chunk = (word >> 2) ^ (row >> 3);       // 16-byte chunk, swizzled
      tile[row * 32 + chunk * 4 + (word & 3)] =
          ptx::pack4_e4m3(f[0][k] * inv_scale, f[1][k] * inv_scale, f[2][k] * inv_scale,
                          f[3][k] * inv_scale);
    }
    __syncthreads();
    // 64 features x 8 chunks of 16 tokens: 512 vectors, two per thread
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int v = threadIdx.x + 256 * i;
      const int row = v >> 3, c = v & 7;
      const int s = s0 + 16 * c;
      if (s < S) {   // S is a multiple of 16: a chunk is either fully inside or outside
        const uint4 r = *reinterpret_cast<const uint4*>(&tile[row * 32 + ((c ^ (row >> 3)) * 4)]);
        *reinterpret_cast<uint4*>(dst + static_cast<long long>(d0 + row) * S + s) = r;
      }
    }
  }
}

int grid_for(long long n, int sms) {
  const long long blocks = (n + 255) / 256;
  const long long cap = static_cast<long long>(sms) * 8;
  return static_cast<int>(blocks < cap ? blocks : cap);
}

}  // namespace

attn_status launch_absmax(const void* in, long long n, bool bf16, float* out,
                          cudaStream_t stream) {
  const int sms = device_sm_count();
  if (sms <= 0) return ATTN_ERR_CUDA;
  if (cudaMemsetAsync(out, 0, sizeof(float), stream) != cudaSuccess) return ATTN_ERR_CUDA;
  const long long n16 = n / 8;
  const int grid = grid_for(n16, sms);
  auto* o = reinterpret_cast<unsigned int*>(out);
  if (bf16)
    absmax_kernel<true><<<grid, 256, 0, stream>>>(static_cast<const uint4*>(in), n16, o);
  else
    absmax_kernel<false><<<grid, 256, 0, stream>>>(static_cast<const uint4*>(in), n16, o);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status launch_quantize_e4m3(const void* in, bool bf16, void* out, int BH, int S, int D,
                                 float inv_scale, bool transpose, cudaStream_t stream) {
  const int sms = device_sm_count();
  if (sms <= 0) return ATTN_ERR_CUDA;
  if (!transpose) {
    const long long n16x2 = static_cast<long long>(BH) * S * D / 16;
    const int grid = grid_for(n16x2, sms);
    if (bf16)
      quantize_kernel<true><<<grid, 256, 0, stream>>>(static_cast<const uint4*>(in),
                                                      static_cast<uint4*>(out), n16x2, inv_scale);
    else
      quantize_kernel<false><<<grid, 256, 0, stream>>>(static_cast<const uint4*>(in),
                                                       static_cast<uint4*>(out), n16x2, inv_scale);
  } else {
    const dim3 grid((S + kTT - 1) / kTT, D / kTF, BH < 65535 ? BH : 65535);
    if (bf16)
      quantize_t_kernel<true><<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(in),
                                                        static_cast<uint8_t*>(out), BH, S, D,
                                                        inv_scale);
    else
      quantize_t_kernel<false><<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(in),
                                                         static_cast<uint8_t*>(out), BH, S, D,
                                                         inv_scale);
  }
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace cpattn
