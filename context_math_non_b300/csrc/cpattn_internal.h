// Internal launchers shared between the C ABI (cpattn_capi.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>

#include "../../include/cpattn.h"

namespace cpattn {

// Default bound on any single wait inside the attention kernel: 2 seconds.
constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;

int device_sm_count();

// Attention over P KV chunks (P = 1: plain attention).  Arguments already validated.
// max_ctas > 0 caps the persistent grid (testing only); 0 = one CTA per SM.  ring = false: one
// partial (O_c, LSE_c) per chunk; ring = true: every query block walks all P chunks in ring
// order keeping its running softmax state on chip, and writes one merged O and LSE.
attn_status launch_attention(const void* q, const void* k, const void* v, void* o, float* lse,
                             int P, int B, int H, int Sq, int Skv, int D, bool bf16, float scale,
                             cudaStream_t stream, unsigned long long limit_ns, int max_ctas,
                             bool ring = false);

// 1: D = 128 attention runs on CTA pairs; 0 (default): single-CTA kernel for every D.
// Returns the previous setting.
int set_attention_variant(int v);

// Ulysses attention reading Q/K/V and writing O in the sequence-sharded layout
// [R][B][S/R][H][D] (R = rank count); LSE in the head-sharded order [R][B][H/R][S].
attn_status launch_attention_ulysses(const void* q, const void* k, const void* v, void* o,
                                     float* lse, int R, int B, int S, int H, int D, bool bf16,
                                     float scale, cudaStream_t stream,
                                     unsigned long long limit_ns, int max_ctas);

// e4m3 attention (D = 128) in ring mode over P chunks: q, k [B*H][S][128] e4m3, vt [B*H][128][Skv]
// e4m3 (V transposed), real value = byte value * the tensor's scale; O bf16 [B*H][Sq][128].
attn_status launch_attention_fp8(const void* q, const void* k, const void* vt, void* o,
                                 float* lse, int P, int B, int H, int Sq, int Skv, float scale,
                                 float q_scale, float k_scale, float v_scale, cudaStream_t stream,
                                 unsigned long long limit_ns, int max_ctas);

// max |x| of n 16-bit elements (n % 8 == 0) into *out (device fp32; zeroed first on `stream`).
attn_status launch_absmax(const void* in, long long n, bool bf16, float* out, cudaStream_t stream);

// y = e4m3(x * inv_scale): [BH][S][D] -> [BH][S][D], or -> [BH][D][S] when transpose.
attn_status launch_quantize_e4m3(const void* in, bool bf16, void* out, int BH, int S, int D,
                                 float inv_scale, bool transpose, cudaStream_t stream);

attn_status launch_lse_merge(const void* o_parts, const float* lse_parts, int P, long long rows,
                             int D, bool bf16, void* o, float* lse, cudaStream_t stream);

attn_status launch_layout(const void* in, void* out, int P, int B, int S, int H, int D,
                          int elem_bytes, bool seq2head, cudaStream_t stream);

attn_status launch_watchdog_selftest(unsigned long long limit_ns, cudaStream_t stream);

attn_status read_and_clear_device_status(cudaStream_t stream);

attn_status launch_mma_probe(int n, int mode, int iters, cudaStream_t stream);

attn_status launch_alu_probe(int mode, int iters, cudaStream_t stream);

}  // namespace cpattn
