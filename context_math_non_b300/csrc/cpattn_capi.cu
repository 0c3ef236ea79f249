// C ABI of the context-parallel attention library: argument validation on the host, then one
// kernel launch per call.  Nothing here touches the GPU before the arguments are known to be
// valid, so an argument error leaves every buffer untouched.

#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>

#include "../../include/cpattn.h"
#include "cpattn_internal.h"

namespace {

std::atomic<int> g_max_ctas{0};

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

// Byte ranges [a, a+na) and [b, b+nb) intersect (empty ranges never do).
bool overlaps(const void* a, long long na, const void* b, long long nb) {
  if (a == nullptr || b == nullptr || na <= 0 || nb <= 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + static_cast<uintptr_t>(nb) && y < x + static_cast<uintptr_t>(na);
}

bool valid_dtype(attn_dtype dt) { return dt == ATTN_BF16 || dt == ATTN_FP16; }

float resolve_scale(float scale, int D) {
  return (scale > 0.f && std::isfinite(scale)) ? scale : 1.0f / std::sqrt(static_cast<float>(D));
}

// Shared checks of attn_fwd / attn_fwd_chunked.  Returns ATTN_OK and sets *empty when there is
// nothing to compute.
attn_status check_attention(const void* q, const void* k, const void* v, const void* o,
                            const float* lse, int P, int B, int H, int Sq, int Skv, int D,
                            attn_dtype dt, bool* empty) {
  *empty = false;
  if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
  if (B < 0 || H < 0 || Sq < 0 || Skv < 1 || D < 1 || !valid_dtype(dt))
    return ATTN_ERR_INVALID_ARG;
  if (P < 1 || P > Skv) return ATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H > INT_MAX) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(o) || misaligned(lse))
    return ATTN_ERR_MISALIGNED;
  if (B == 0 || H == 0 || Sq == 0) {
    *empty = true;
    return ATTN_OK;
  }
  const long long bh = static_cast<long long>(B) * H;
  const long long qbytes = bh * Sq * D * 2, kvbytes = bh * Skv * D * 2;
  const long long obytes = qbytes * P, lbytes = bh * Sq * 4 * P;
  for (const void* in : {q, k, v}) {
    const long long n = in == q ? qbytes : kvbytes;
    if (overlaps(o, obytes, in, n) || overlaps(lse, lbytes, in, n)) return ATTN_ERR_INVALID_ARG;
  }
  if (overlaps(o, obytes, lse, lbytes)) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

attn_status check_layout(const void* in, const void* out, int P, int B, int S, int H, int D,
                         int elem_bytes, bool* empty) {
  *empty = false;
  if (!in || !out) return ATTN_ERR_INVALID_ARG;
  if (P < 1 || B < 0 || S < 0 || H < 0 || D < 1 || elem_bytes < 1) return ATTN_ERR_INVALID_ARG;
  if (S % P != 0 || H % P != 0) return ATTN_ERR_INVALID_ARG;
  if ((static_cast<long long>(D) * elem_bytes) % 16 != 0) return ATTN_ERR_INVALID_ARG;
  if (misaligned(in) || misaligned(out)) return ATTN_ERR_MISALIGNED;
  const long long bytes = static_cast<long long>(B) * S * H * D * elem_bytes;
  if (bytes == 0) {
    *empty = true;
    return ATTN_OK;
  }
  if (overlaps(in, bytes, out, bytes)) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

}  // namespace

extern "C" {

attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int Sq, int Skv, int D, attn_dtype dt, float scale,
                     attn_stream_t stream) {
  bool empty;
  attn_status st = check_attention(q, k, v, o, lse, 1, B, H, Sq, Skv, D, dt, &empty);
  if (st != ATTN_OK || empty) return st;
  return cpattn::launch_attention(q, k, v, o, lse, 1, B, H, Sq, Skv, D, dt == ATTN_BF16,
                                  resolve_scale(scale, D), reinterpret_cast<cudaStream_t>(stream),
                                  cpattn::kDefaultWaitLimitNs, g_max_ctas.load());
}

attn_status attn_fwd_chunked(const void* q, const void* k, const void* v, int P, void* o_parts,
                             float* lse_parts, int B, int H, int Sq, int Skv, int D,
                             attn_dtype dt, float scale, attn_stream_t stream) {
  if (lse_parts == nullptr) return ATTN_ERR_INVALID_ARG;
  bool empty;
  attn_status st = check_attention(q, k, v, o_parts, lse_parts, P, B, H, Sq, Skv, D, dt, &empty);
  if (st != ATTN_OK || empty) return st;
  return cpattn::launch_attention(q, k, v, o_parts, lse_parts, P, B, H, Sq, Skv, D,
                                  dt == ATTN_BF16, resolve_scale(scale, D),
                                  reinterpret_cast<cudaStream_t>(stream),
                                  cpattn::kDefaultWaitLimitNs, g_max_ctas.load());
}

attn_status attn_fwd_ring(const void* q, const void* k, const void* v, int P, void* o, float* lse,
                          int B, int H, int Sq, int Skv, int D, attn_dtype dt, float scale,
                          attn_stream_t stream) {
  bool empty;
  // O and LSE are single outputs here: validate them as the P = 1 problem, then check P alone.
  attn_status st = check_attention(q, k, v, o, lse, 1, B, H, Sq, Skv, D, dt, &empty);
  if (st != ATTN_OK) return st;
  if (P < 1 || P > Skv) return ATTN_ERR_INVALID_ARG;
  if (empty) return ATTN_OK;
  return cpattn::launch_attention(q, k, v, o, lse, P, B, H, Sq, Skv, D, dt == ATTN_BF16,
                                  resolve_scale(scale, D), reinterpret_cast<cudaStream_t>(stream),
                                  cpattn::kDefaultWaitLimitNs, g_max_ctas.load(), true);
}

attn_status attn_fwd_ulysses(const void* q, const void* k, const void* v, void* o, float* lse,
                             int P, int B, int S, int H, int D, attn_dtype dt, float scale,
                             attn_stream_t stream) {
  if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
  if (P < 1 || B < 0 || S < 0 || H < 0 || D < 1 || !valid_dtype(dt)) return ATTN_ERR_INVALID_ARG;
  if (S % P != 0 || H % P != 0) return ATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H > INT_MAX) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(o) || misaligned(lse))
    return ATTN_ERR_MISALIGNED;
  if (B == 0 || H == 0 || S == 0) return ATTN_OK;
  if ((S / P) % 16 != 0) return ATTN_ERR_UNSUPPORTED;
  const long long bytes = static_cast<long long>(B) * S * H * D * 2;
  const long long lbytes = static_cast<long long>(B) * S * H * 4;
  for (const void* in : {q, k, v})
    if (overlaps(o, bytes, in, bytes) || overlaps(lse, lbytes, in, bytes))
      return ATTN_ERR_INVALID_ARG;
  if (overlaps(o, bytes, lse, lbytes)) return ATTN_ERR_INVALID_ARG;
  return cpattn::launch_attention_ulysses(q, k, v, o, lse, P, B, S, H, D, dt == ATTN_BF16,
                                          resolve_scale(scale, D),
                                          reinterpret_cast<cudaStream_t>(stream),
                                          cpattn::kDefaultWaitLimitNs, g_max_ctas.load());
}

attn_status attn_fwd_fp8(const void* q, const void* k, const void* vt, int P, float q_scale,
                         float k_scale, float v_scale, void* o, float* lse, int B, int H, int Sq,
                         int Skv, int D, float scale, attn_stream_t stream) {
  if (!q || !k || !vt || !o) return ATTN_ERR_INVALID_ARG;
  if (B < 0 || H < 0 || Sq < 0 || Skv < 1 || D < 1) return ATTN_ERR_INVALID_ARG;
  if (P < 1 || P > Skv) return ATTN_ERR_INVALID_ARG;
  for (float sc : {q_scale, k_scale, v_scale})
    if (!(sc > 0.f) || !std::isfinite(sc)) return ATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H > INT_MAX) return ATTN_ERR_INVALID_ARG;
  if (D != 128) return ATTN_ERR_UNSUPPORTED;
  // V^T rows are Skv bytes long and every KV tile starts at a multiple of 16 keys (the TMA
  // alignment of one-byte elements): chunks must be equal and a multiple of 16 keys.
  if (Skv % 16 != 0) return ATTN_ERR_UNSUPPORTED;
  if (P > 1 && (Skv % P != 0 || (Skv / P) % 16 != 0)) return ATTN_ERR_UNSUPPORTED;
  if (misaligned(q) || misaligned(k) || misaligned(vt) || misaligned(o) || misaligned(lse))
    return ATTN_ERR_MISALIGNED;
  if (B == 0 || H == 0 || Sq == 0) return ATTN_OK;
  const long long bh = static_cast<long long>(B) * H;
  const long long qbytes = bh * Sq * D, kvbytes = bh * Skv * D;
  const long long obytes = qbytes * 2, lbytes = bh * Sq * 4;
  for (const void* in : {q, k, vt}) {
    const long long n = in == q ? qbytes : kvbytes;
    if (overlaps(o, obytes, in, n) || overlaps(lse, lbytes, in, n)) return ATTN_ERR_INVALID_ARG;
  }
  if (overlaps(o, obytes, lse, lbytes)) return ATTN_ERR_INVALID_ARG;
  return cpattn::launch_attention_fp8(q, k, vt, o, lse, P, B, H, Sq, Skv,
                                      resolve_scale(scale, D), q_scale, k_scale, v_scale,
                                      reinterpret_cast<cudaStream_t>(stream),
                                      cpattn::kDefaultWaitLimitNs, g_max_ctas.load());
}

attn_status cp_absmax(const void* x, long long n, attn_dtype dt, float* amax,
                      attn_stream_t stream) {
  if (!x || !amax || n < 0 || !valid_dtype(dt)) return ATTN_ERR_INVALID_ARG;
  if (n % 8 != 0) return ATTN_ERR_INVALID_ARG;
  if (misaligned(x) || (reinterpret_cast<uintptr_t>(amax) & 3u) != 0) return ATTN_ERR_MISALIGNED;
  if (overlaps(amax, 4, x, n * 2)) return ATTN_ERR_INVALID_ARG;
  return cpattn::launch_absmax(x, n, dt == ATTN_BF16, amax,
                               reinterpret_cast<cudaStream_t>(stream));
}

attn_status cp_quantize_e4m3(const void* x, attn_dtype dt, void* y, int BH, int S, int D,
                             float scale, int transpose, attn_stream_t stream) {
  if (!x || !y || BH < 0 || S < 0 || D < 1 || !valid_dtype(dt)) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (D % 16 != 0) return ATTN_ERR_INVALID_ARG;
  if (transpose && (D % 64 != 0 || S % 16 != 0)) return ATTN_ERR_INVALID_ARG;
  if (misaligned(x) || misaligned(y)) return ATTN_ERR_MISALIGNED;
  const long long n = static_cast<long long>(BH) * S * D;
  if (n == 0) return ATTN_OK;
  if (overlaps(x, n * 2, y, n)) return ATTN_ERR_INVALID_ARG;
  const float inv = 1.0f / scale;
  if (!std::isfinite(inv)) return ATTN_ERR_INVALID_ARG;
  return cpattn::launch_quantize_e4m3(x, dt == ATTN_BF16, y, BH, S, D, inv, transpose != 0,
                                      reinterpret_cast<cudaStream_t>(stream));
}

attn_status attn_lse_merge(const void* o_parts, const float* lse_parts, int P, int B, int H,
                           int Sq, int D, attn_dtype dt, void* o, float* lse,
                           attn_stream_t stream) {
  if (!o_parts || !lse_parts || !o) return ATTN_ERR_INVALID_ARG;
  if (P < 1 || B < 0 || H < 0 || Sq < 0 || D < 1 || !valid_dtype(dt)) return ATTN_ERR_INVALID_ARG;
  if ((D * 2) % 16 != 0) return ATTN_ERR_INVALID_ARG;
  if (misaligned(o_parts) || misaligned(lse_parts) || misaligned(o) || misaligned(lse))
    return ATTN_ERR_MISALIGNED;
  const long long rows = static_cast<long long>(B) * H * Sq;
  if (rows == 0) return ATTN_OK;
  const long long pbytes = rows * D * 2 * P, plbytes = rows * 4 * P;
  const long long obytes = rows * D * 2, lbytes = rows * 4;
  if (overlaps(o, obytes, o_parts, pbytes) || overlaps(o, obytes, lse_parts, plbytes) ||
      overlaps(lse, lbytes, o_parts, pbytes) || overlaps(lse, lbytes, lse_parts, plbytes) ||
      overlaps(o, obytes, lse, lbytes))
    return ATTN_ERR_INVALID_ARG;
  return cpattn::launch_lse_merge(o_parts, lse_parts, P, rows, D, dt == ATTN_BF16, o, lse,
                                  reinterpret_cast<cudaStream_t>(stream));
}

attn_status cp_layout_seq2head(const void* in, void* out, int P, int B, int S, int H, int D,
                               int elem_bytes, attn_stream_t stream) {
  bool empty;
  attn_status st = check_layout(in, out, P, B, S, H, D, elem_bytes, &empty);
  if (st != ATTN_OK || empty) return st;
  return cpattn::launch_layout(in, out, P, B, S, H, D, elem_bytes, true,
                               reinterpret_cast<cudaStream_t>(stream));
}

attn_status cp_layout_head2seq(const void* in, void* out, int P, int B, int S, int H, int D,
                               int elem_bytes, attn_stream_t stream) {
  bool empty;
  attn_status st = check_layout(in, out, P, B, S, H, D, elem_bytes, &empty);
  if (st != ATTN_OK || empty) return st;
  return cpattn::launch_layout(in, out, P, B, S, H, D, elem_bytes, false,
                               reinterpret_cast<cudaStream_t>(stream));
}

const char* attn_status_string(attn_status status) {
  switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_MISALIGNED: return "ATTN_ERR_MISALIGNED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
  }
  return "ATTN_ERR_UNKNOWN";
}

attn_status attn_device_status(attn_stream_t stream) {
  return cpattn::read_and_clear_device_status(reinterpret_cast<cudaStream_t>(stream));
}

attn_status attn_watchdog_selftest(uint64_t limit_ns, attn_stream_t stream) {
  if (limit_ns < 1000ull) limit_ns = 1000ull;
  if (limit_ns > 10000000000ull) limit_ns = 10000000000ull;
  return cpattn::launch_watchdog_selftest(limit_ns, reinterpret_cast<cudaStream_t>(stream));
}

attn_status attn_probe_mma(int n, int mode, int iters, attn_stream_t stream) {
  if ((n != 64 && n != 128 && n != 256) || mode < 0 || mode > 10 || iters < 1)
    return ATTN_ERR_INVALID_ARG;
  if (mode >= 2 && n != 128) return ATTN_ERR_INVALID_ARG;
  return cpattn::launch_mma_probe(n, mode, iters, reinterpret_cast<cudaStream_t>(stream));
}

attn_status attn_probe_alu(int mode, int iters, attn_stream_t stream) {
  if (mode < 0 || mode > 5 || iters < 1) return ATTN_ERR_INVALID_ARG;
  return cpattn::launch_alu_probe(mode, iters, reinterpret_cast<cudaStream_t>(stream));
}

int attn_set_kernel_variant(int v) { return cpattn::set_attention_variant(v != 0 ? 1 : 0); }

int attn_set_max_ctas(int n) { return g_max_ctas.exchange(n > 0 ? n : 0); }

int attn_version(void) { return 100; }

}  // extern "C"
