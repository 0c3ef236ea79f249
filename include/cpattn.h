/*
 * cpattn.h -- C ABI of the context-parallel attention primitives for B300 (sm_103a).
 *
 * The operations are those of context-parallel inference for diffusion transformers as described
 * on "Scaling AI Inference Across Multiple GPUs Using NVIDIA TensorRT with Multi-Device Inference
 * Support", section "Parallelism strategies for distributed inference" (subsections "Context
 * parallelism", "Ring Attention", "DeepSpeed Ulysses").  One GPU stands in for P ranks: a ring
 * step becomes one KV chunk, and the Ulysses all-to-all becomes an on-device re-layout.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The library allocates no device
 *    memory.  Inputs are never written.  Outputs must not overlap inputs.
 *  - Tensors are dense and row-major in the order given in brackets (last index contiguous).
 *  - Every tensor pointer must be 16-byte aligned (ATTN_ERR_MISALIGNED otherwise).
 *  - Calls are asynchronous on `stream` (NULL = the legacy default stream).  They return after
 *    the launch.  Argument errors are detected on the host before anything is launched, and then
 *    nothing is written.  A failed launch returns ATTN_ERR_CUDA.
 *  - Zero-sized batch / head / query / sequence extents are accepted and launch nothing.
 *  - The compute calls are thread-safe and may run concurrently on different streams and
 *    devices (the one-time kernel set-up is done per device).  The only device-side state is
 *    one status word per device, written by the attention kernels' watchdog and shared by every
 *    stream and call on that device (see attn_device_status).  attn_set_max_ctas and
 *    attn_set_kernel_variant are process-wide test and measurement switches: a launch on
 *    another thread sees either the old or the new setting.
 *  - 16-bit types are IEEE fp16 or bfloat16; LSE values are fp32 natural logarithms.
 */
#ifndef CPATTN_H
#define CPATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CPATTN_API __attribute__((visibility("default")))
#else
#define CPATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream, declared without the CUDA headers. */
typedef struct CUstream_st* attn_stream_t;

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,  /* null pointer, bad extent, P out of range, overlapping buffers  */
  ATTN_ERR_UNSUPPORTED = 2,  /* valid request the kernels do not implement (e.g. D not 64/128) */
  ATTN_ERR_MISALIGNED = 3,   /* a pointer is not 16-byte aligned                                */
  ATTN_ERR_CUDA = 4,         /* a CUDA runtime / driver call failed                             */
  ATTN_ERR_TIMEOUT = 5       /* a kernel's bounded wait expired (reported by attn_device_status) */
} attn_status;

typedef enum { ATTN_BF16 = 0, ATTN_FP16 = 1 } attn_dtype;

/*
 * attn_fwd -- non-causal multi-head attention forward.
 *   Defines: page section "Context parallelism" (bidirectional attention of a diffusion
 *   transformer over the whole sequence): O = softmax(Q K^T * scale) V.
 *   q   [B][H][Sq][D]   dtype `dt`
 *   k,v [B][H][Skv][D]  dtype `dt`
 *   o   [B][H][Sq][D]   dtype `dt`, written (fp32 accumulation, rounded to nearest even)
 *   lse [B][H][Sq] fp32, written if non-NULL: ln sum_j exp(scale * q.k_j)
 *   D must be 64 or 128 (ATTN_ERR_UNSUPPORTED otherwise); Skv >= 1.
 *   scale <= 0 selects 1/sqrt(D).
 */
CPATTN_API attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int H, int Sq, int Skv, int D, attn_dtype dt, float scale,
                     attn_stream_t stream);

/*
 * attn_fwd_chunked -- per-KV-chunk partial outputs (one ring step per chunk).
 *   Defines: page subsection "Ring Attention" and Figure 3: each rank holds a slice of K and V,
 *   and the attention output is built up slice by slice with an online softmax.
 *   KV rows are split into P contiguous chunks; chunk c covers rows
 *   [floor(c*Skv/P), floor((c+1)*Skv/P)).  For each chunk the kernel writes the attention of Q
 *   over that chunk only, normalised over the chunk, and its LSE:
 *   o_parts   [P][B][H][Sq][D]  dtype `dt`
 *   lse_parts [P][B][H][Sq]     fp32 (required)
 *   attn_lse_merge of these partials reproduces attn_fwd.  1 <= P <= Skv; other arguments as
 *   for attn_fwd.
 *   Short chunks cost throughput here: every chunk ends with a normalised partial output of
 *   the full query length (P times the bytes of O) and an accumulator drain, e.g. ~0.76 of the
 *   P = 1 rate at 576-key chunks.  When only the merged result is wanted, attn_fwd_ring
 *   computes it with the running state kept on chip across chunks (~0.84 of the P = 1 rate at
 *   576-key chunks, where the masked half tile at each chunk end is the remaining cost).
 */
CPATTN_API attn_status attn_fwd_chunked(const void* q, const void* k, const void* v, int P,
                             void* o_parts, float* lse_parts,
                             int B, int H, int Sq, int Skv, int D, attn_dtype dt, float scale,
                             attn_stream_t stream);

/*
 * attn_lse_merge -- combine P partial attention outputs by their log-sum-exp.
 *   Defines: page subsection "Ring Attention" (the output is updated as each KV block streams
 *   past).  Per row, with M = max_c LSE_c and w_c = exp(LSE_c - M):
 *     O = sum_c w_c O_c / sum_c w_c,  LSE = M + ln sum_c w_c.
 *   A row whose partials all have LSE = -inf merges to O = 0, LSE = -inf.
 *   o_parts   [P][B][H][Sq][D] dtype `dt`;  lse_parts [P][B][H][Sq] fp32
 *   o         [B][H][Sq][D]    dtype `dt`;  lse [B][H][Sq] fp32, written if non-NULL
 *   P >= 1; D >= 1 with D * 2 bytes a multiple of 16.
 */
CPATTN_API attn_status attn_lse_merge(const void* o_parts, const float* lse_parts, int P,
                           int B, int H, int Sq, int D, attn_dtype dt,
                           void* o, float* lse, attn_stream_t stream);

/*
 * cp_layout_seq2head -- the first DeepSpeed Ulysses all-to-all, as one on-device re-layout.
 *   Defines: page subsection "DeepSpeed Ulysses" and Figure 4: sequence sharding becomes head
 *   sharding, every rank then holding the full sequence for a disjoint subset of heads.
 *   in  [P][B][S/P][H][D]   rank p holds tokens p*S/P .. (p+1)*S/P-1, all heads
 *   out [P][B][H/P][S][D]   rank g holds all tokens (global order), heads g*H/P .. (g+1)*H/P-1
 *   out[g][b][j][p*S/P + s][d] = in[p][b][s][g*H/P + j][d]  (bit copy of elem_bytes each)
 *   Requires P >= 1, S % P == 0, H % P == 0, (D * elem_bytes) % 16 == 0, no overlap.
 */
CPATTN_API attn_status cp_layout_seq2head(const void* in, void* out, int P, int B, int S, int H, int D,
                               int elem_bytes, attn_stream_t stream);

/*
 * cp_layout_head2seq -- the second Ulysses all-to-all: exact inverse of cp_layout_seq2head.
 *   Defines: page subsection "DeepSpeed Ulysses" (results gathered across heads and
 *   re-partitioned along the sequence).
 *   in  [P][B][H/P][S][D] -> out [P][B][S/P][H][D]; same requirements.
 */
CPATTN_API attn_status cp_layout_head2seq(const void* in, void* out, int P, int B, int S, int H, int D,
                               int elem_bytes, attn_stream_t stream);

/*
 * attn_fwd_ring -- Ring Attention with the merge fused into the attention kernel.
 *   Defines: page section "Ring Attention" (Figure 3) -- each rank keeps its query block, the
 *   KV blocks travel around the ring, and after every step the rank updates its attention
 *   output with the block it just received.  Here rank c's KV block is chunk c of K/V (chunk
 *   bounds as in attn_fwd_chunked) and the query rows are split into P ranks the same way; each
 *   block of 256 query rows starts at the chunk of the rank that holds its first row and then
 *   takes the chunks c-1, c-2, ... (mod P), every chunk cut into 128-row tiles from its own first
 *   row (last tile masked at the chunk end).  The running max, denominator and output stay on
 *   chip across chunks, so no partial output reaches memory and no merge pass runs.  Result:
 *   full attention over Skv keys, equal to attn_lse_merge(attn_fwd_chunked(P)) and to attn_fwd
 *   up to fp32 summation order.
 *   q [B][H][Sq][D], k, v [B][H][Skv][D] dtype `dt`; o [B][H][Sq][D]; lse [B][H][Sq] fp32 or NULL.
 *   1 <= P <= Skv (ATTN_ERR_INVALID_ARG otherwise); other requirements as attn_fwd.
 */
CPATTN_API attn_status attn_fwd_ring(const void* q, const void* k, const void* v, int P, void* o,
                                     float* lse, int B, int H, int Sq, int Skv, int D,
                                     attn_dtype dt, float scale, attn_stream_t stream);

/*
 * attn_fwd_fp8 -- attention on e4m3 inputs with per-tensor scales (the 8-bit variant the pages
 *   recommend for attention layers: page section on quantisation, "FP8 for attention").
 *   Real inputs are q_scale*Q8, k_scale*K8, v_scale*V8.  S = Q8 K8^T and O = P8 V8 run on the
 *   tensor cores in e4m3 with fp32 accumulation; the softmax is fp32 (logits times
 *   scale*q_scale*k_scale); the softmax weights P are rounded to e4m3 (values in [0, 256],
 *   round to nearest even) for the P*V product, while the denominator sums the fp32 weights.
 *   The KV sequence is walked in P chunks in ring order exactly as attn_fwd_ring (P = 1: plain
 *   attention).  Output O in bf16, O = v_scale * (P8 V8) / l.
 *   q [B][H][Sq][D], k [B][H][Skv][D] e4m3 bytes; vt [B][H][D][Skv] e4m3 bytes (V transposed,
 *   as cp_quantize_e4m3 with transpose = 1 writes it); o [B][H][Sq][D] bf16; lse [B][H][Sq]
 *   fp32 or NULL (natural log of the sum of exp of the real scaled logits).
 *   D = 128 and Skv % 16 == 0, and for P > 1 equal chunks of a multiple of 16 keys (Skv % P == 0,
 *   (Skv/P) % 16 == 0): ATTN_ERR_UNSUPPORTED otherwise.  Scales must be positive and finite.
 */
CPATTN_API attn_status attn_fwd_fp8(const void* q, const void* k, const void* vt, int P,
                                    float q_scale, float k_scale, float v_scale, void* o,
                                    float* lse, int B, int H, int Sq, int Skv, int D, float scale,
                                    attn_stream_t stream);

/*
 * cp_absmax -- *amax = max |x| over n bf16/fp16 elements (n % 8 == 0; x 16-byte aligned;
 *   amax a device fp32, 4-byte aligned, zeroed by this call before the reduction).  For picking
 *   an e4m3 scale (e.g. amax / 448).  Not part of the paper's method: input preparation for
 *   attn_fwd_fp8.
 */
CPATTN_API attn_status cp_absmax(const void* x, long long n, attn_dtype dt, float* amax,
                                 attn_stream_t stream);

/*
 * cp_quantize_e4m3 -- y = e4m3(x * (1/scale)), fp32 multiply, round to nearest even, saturating
 *   to +-448 (NaN stays NaN).  x [BH][S][D] bf16/fp16; y [BH][S][D] bytes (transpose = 0) or
 *   [BH][D][S] (transpose = 1, the V layout attn_fwd_fp8 takes).  D % 16 == 0; transposed:
 *   D % 64 == 0 and S % 16 == 0 (ATTN_ERR_INVALID_ARG otherwise).  Input preparation for
 *   attn_fwd_fp8.
 */
CPATTN_API attn_status cp_quantize_e4m3(const void* x, attn_dtype dt, void* y, int BH, int S,
                                        int D, float scale, int transpose, attn_stream_t stream);

/*
 * attn_fwd_ulysses -- DeepSpeed Ulysses attention without the two re-layout passes.
 *   Defines: page subsection "DeepSpeed Ulysses" and Figure 4 -- after the first all-to-all each
 *   rank attends over the full sequence for its subset of heads, and the second all-to-all
 *   returns the output to sequence sharding.  Here both all-to-alls are folded into the
 *   attention kernel's addressing: Q, K, V are read and O is written in the sequence-sharded
 *   layout, and the result equals
 *     cp_layout_head2seq(attn_fwd(cp_layout_seq2head(q), cp_layout_seq2head(k),
 *                                 cp_layout_seq2head(v)))  (attention per head, full sequence).
 *   q, k, v, o [P][B][S/P][H][D]  dtype `dt`   (rank p holds tokens p*S/P .. (p+1)*S/P - 1)
 *   lse        [P][B][H/P][S] fp32, written if non-NULL (rank g, batch b, head g*H/P + j, token t)
 *   Requires S % P == 0, H % P == 0, (S/P) % 16 == 0 (ATTN_ERR_UNSUPPORTED otherwise: token tiles
 *   are gathered in boxes that never straddle two ranks' shards), D = 64 or 128.
 */
CPATTN_API attn_status attn_fwd_ulysses(const void* q, const void* k, const void* v, void* o,
                                        float* lse, int P, int B, int S, int H, int D,
                                        attn_dtype dt, float scale, attn_stream_t stream);

/* Human-readable name of a status code (static string, never NULL). */
CPATTN_API const char* attn_status_string(attn_status status);

/*
 * attn_device_status -- synchronise `stream`, then return and clear the device status word.
 *   The attention kernels bound every internal wait; a wait that expires records
 *   ATTN_ERR_TIMEOUT there and the kernel returns early instead of hanging (its outputs are then
 *   undefined).  Returns ATTN_OK if nothing was recorded, ATTN_ERR_CUDA if the synchronisation
 *   itself failed.
 */
CPATTN_API attn_status attn_device_status(attn_stream_t stream);

/*
 * attn_watchdog_selftest -- launch one block that waits, with the attention kernels' bounded
 *   wait, on a barrier that nothing ever signals, giving up after `limit_ns` nanoseconds
 *   (clamped to [1e3, 1e10]).  The expected outcome is that attn_device_status then reports
 *   ATTN_ERR_TIMEOUT.  Exists so the failure path can be tested without faulting a GPU.
 */
CPATTN_API attn_status attn_watchdog_selftest(uint64_t limit_ns, attn_stream_t stream);

/*
 * attn_set_max_ctas -- cap the persistent attention grid at `n` CTAs (n <= 0 restores the
 *   default of one CTA per SM).  Process-wide; affects launches made after the call.  Used to
 *   exercise the many-units-per-CTA path on small problems and to study load balance.  Returns
 *   the previous cap.
 */
CPATTN_API int attn_set_max_ctas(int n);

/*
 * attn_probe_mma -- tensor-core ceiling probe (calibration, no data movement).
 *   One CTA per SM issues `iters` tcgen05.mma kind::f16 instructions back to back: M = 128,
 *   N = n (64, 128 or 256), K = 16, bf16 operands, fp32 accumulation in tensor memory.
 *   mode 0: A and B from shared memory (the S = Q K^T form); mode 1: A from tensor memory (the
 *   O += P V form); mode 2 (n = 128 only): the attention kernel's per-KV-step sequence of four
 *   GEMMs with a commit after each, iters/32 steps; mode 3: as mode 2 with a
 *   tcgen05.fence::after_thread_sync before each P*V GEMM; mode 4 (n = 128): iters/8 serial
 *   round trips of one 128x128x128 GEMM -> commit -> a second warp waits, reads tensor memory
 *   and arrives -> the issuing thread waits (hand-off latency); modes 5 / 6 / 7 (n = 128): mode
 *   2 while four other warps stream tensor-memory loads and stores / run dependent FMA chains /
 *   run independent FMA chains (contention); mode 8 (n = 128): the D = 64 per-step sequence
 *   (per query tile 8 A-from-tensor-memory MMAs with N = 64, then 4 shared-memory MMAs with
 *   N = 128, one commit; two tiles) issued by a single lane, iters/24 steps; mode 9: the same
 *   issued by a converged warp through elect.sync; mode 10: the D = 128 sequence of mode 2
 *   issued through elect.sync, iters/32 steps.  The caller times the launch:
 *   flops = SMs * iters * 2*128*n*16 for modes 0-7, SMs * steps * 2 * 4*128*128*D for 8-10.
 *   ATTN_ERR_INVALID_ARG for other arguments.
 */
CPATTN_API attn_status attn_probe_mma(int n, int mode, int iters, attn_stream_t stream);

/*
 * attn_probe_alu -- throughput probe of the softmax's instruction mix (calibration).
 *   2 blocks of 512 threads per SM; every thread runs 8 independent dependent chains of one
 *   operation for `iters` iterations.  mode 0: ex2.approx.ftz.f32 (MUFU); 1: cvt.rn.bf16x2.f32;
 *   2: fma.rn.f32x2 (one pair per op); 3: fma.rn.f32; 4: ex2.approx.ftz.bf16x2 and
 *   5: ex2.approx.f16x2 (two exponentials per op).  The caller times the launch:
 *   ops = SMs * 2 * 512 * iters * 8.  ATTN_ERR_INVALID_ARG for other modes or iters < 1.
 */
CPATTN_API attn_status attn_probe_alu(int mode, int iters, attn_stream_t stream);

/*
 * attn_set_kernel_variant -- choose the attention kernel for D = 128 (process-wide, affects later
 *   launches): 0 (default) runs the single-CTA kernel; 1 runs it on pairs of SMs (cta_group::2
 *   MMAs, each CTA loading half of every K/V tile -- measured slower on B300, kept for testing
 *   and measurement).  D = 64 always uses the single-CTA kernel.  Both produce results within
 *   the same tolerance.  Returns the previous setting.
 */
CPATTN_API int attn_set_kernel_variant(int v);

/* Library version: major * 10000 + minor * 100 + patch. */
CPATTN_API int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CPATTN_H */
