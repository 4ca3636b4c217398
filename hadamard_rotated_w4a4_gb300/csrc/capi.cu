// extern "C" entry points of libw4a4.so (declared in include/w4a4.h): argument
// checks, operand tags, status codes and the thread-local error message.  No
// entry point allocates memory, throws or aborts.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "../../include/w4a4.h"
#include "w4a4_kernels.cuh"

namespace w4a4 {

int num_sms() {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev < 64) cache[dev] = n;
  return n;
}

}  // namespace w4a4

namespace {

thread_local char g_err[512] = "";

w4a4_status fail(w4a4_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

w4a4_status ok() {
  g_err[0] = '\0';
  return W4A4_OK;
}

w4a4_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return ok();
  return fail(W4A4_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round16(size_t x) { return (x + 15) & ~size_t(15); }

bool valid_k(int64_t K) { return K > 0 && K % 32 == 0 && K <= (int64_t(1) << 30); }

w4a4_status check_k_rows(int64_t rows, int64_t K, const char* fn) {
  if (!valid_k(K)) return fail(W4A4_ERR_INVALID_ARG, "%s: K=%lld must be a positive multiple of 32", fn, (long long)K);
  if (rows < 0 || rows > (int64_t(1) << 31)) return fail(W4A4_ERR_INVALID_ARG, "%s: bad row count %lld", fn, (long long)rows);
  return W4A4_OK;
}

w4a4_status check_q4_0(const w4a4_q4_0* w, const char* fn) {
  if (!w) return fail(W4A4_ERR_INVALID_ARG, "%s: weight descriptor is NULL", fn);
  if ((w->tag & W4A4_TAG_MAGIC_MASK) != W4A4_TAG_Q4_0)
    return fail(W4A4_ERR_INVALID_ARG, "%s: weight descriptor tag 0x%08x is not a Q4_0 tag", fn, w->tag);
  w4a4_status s = check_k_rows(w->rows, w->K, fn);
  if (s != W4A4_OK) return s;
  if (w->rows > 0 && (!w->codes || !w->scales || !w->sums))
    return fail(W4A4_ERR_INVALID_ARG, "%s: weight pointers are NULL", fn);
  if (!aligned16(w->codes) || !aligned16(w->scales) || !aligned16(w->sums) || !aligned16(w->expanded))
    return fail(W4A4_ERR_ALIGNMENT, "%s: weight codes/scales/sums/expanded must be 16-byte aligned", fn);
  return W4A4_OK;
}

w4a4_status check_act4(const w4a4_act4* a, const char* fn) {
  if (!a) return fail(W4A4_ERR_INVALID_ARG, "%s: activation descriptor is NULL", fn);
  if ((a->tag & W4A4_TAG_MAGIC_MASK) != W4A4_TAG_ACT4)
    return fail(W4A4_ERR_INVALID_ARG, "%s: activation descriptor tag 0x%08x is not an int4 tag", fn, a->tag);
  w4a4_status s = check_k_rows(a->rows, a->K, fn);
  if (s != W4A4_OK) return s;
  if (a->rows > 0 && (!a->codes || !a->scales))
    return fail(W4A4_ERR_INVALID_ARG, "%s: activation pointers are NULL", fn);
  if (!aligned16(a->codes) || !aligned16(a->scales) || !aligned16(a->expanded))
    return fail(W4A4_ERR_ALIGNMENT, "%s: activation codes/scales/expanded must be 16-byte aligned", fn);
  return W4A4_OK;
}

w4a4_status check_act8(const w4a4_act8* a, const char* fn) {
  if (!a) return fail(W4A4_ERR_INVALID_ARG, "%s: activation descriptor is NULL", fn);
  if ((a->tag & W4A4_TAG_MAGIC_MASK) != W4A4_TAG_ACT8)
    return fail(W4A4_ERR_INVALID_ARG, "%s: activation descriptor tag 0x%08x is not an int8 tag", fn, a->tag);
  w4a4_status s = check_k_rows(a->rows, a->K, fn);
  if (s != W4A4_OK) return s;
  if (a->rows > 0 && (!a->codes || !a->scales))
    return fail(W4A4_ERR_INVALID_ARG, "%s: activation pointers are NULL", fn);
  if (!aligned16(a->codes) || !aligned16(a->scales))
    return fail(W4A4_ERR_ALIGNMENT, "%s: activation codes/scales must be 16-byte aligned", fn);
  return W4A4_OK;
}

w4a4_status check_act16(const w4a4_act16* a, const char* fn) {
  if (!a) return fail(W4A4_ERR_INVALID_ARG, "%s: activation descriptor is NULL", fn);
  if ((a->tag & W4A4_TAG_MAGIC_MASK) != W4A4_TAG_ACT16)
    return fail(W4A4_ERR_INVALID_ARG, "%s: activation descriptor tag 0x%08x is not a bf16 tag", fn, a->tag);
  w4a4_status s = check_k_rows(a->rows, a->K, fn);
  if (s != W4A4_OK) return s;
  if (a->rows > 0 && !a->values) return fail(W4A4_ERR_INVALID_ARG, "%s: activation values are NULL", fn);
  if (!aligned16(a->values)) return fail(W4A4_ERR_ALIGNMENT, "%s: activation values must be 16-byte aligned", fn);
  return W4A4_OK;
}

template <class A>
w4a4_status check_pair(const w4a4_q4_0* w, const A* a, const char* fn) {
  if (w->K != a->K)
    return fail(W4A4_ERR_MISMATCH, "%s: weights have K=%lld, activations K=%lld", fn, (long long)w->K, (long long)a->K);
  if ((w->tag & W4A4_TAG_ROTATED) != (a->tag & W4A4_TAG_ROTATED))
    return fail(W4A4_ERR_MISMATCH, "%s: weights are %s but activations are %s; refusing a product that would be "
                "silently wrong", fn, (w->tag & W4A4_TAG_ROTATED) ? "H32-rotated" : "unrotated",
                (a->tag & W4A4_TAG_ROTATED) ? "H32-rotated" : "unrotated");
  return W4A4_OK;
}

}  // namespace

extern "C" {

size_t w4a4_q4_0_codes_bytes(int64_t rows, int64_t K) {
  if (!valid_k(K) || rows < 0) return 0;
  return static_cast<size_t>(rows) * static_cast<size_t>(K / 2);
}
size_t w4a4_q4_0_scales_bytes(int64_t rows, int64_t K) {
  if (!valid_k(K) || rows < 0) return 0;
  // padded to 16 bytes: the GEMM reads each fp16 scale through its aligned 4-byte word
  return round16(static_cast<size_t>(rows) * static_cast<size_t>(K / 32) * 2);
}
size_t w4a4_q4_0_sums_bytes(int64_t rows, int64_t K) { return w4a4_q4_0_scales_bytes(rows, K); }
size_t w4a4_q4_0_expanded_bytes(int64_t rows, int64_t K) {
  if (!valid_k(K) || rows < 0) return 0;
  return round16(static_cast<size_t>((rows + 7) / 8 * 8) * static_cast<size_t>(K));
}
size_t w4a4_act4_codes_bytes(int64_t rows, int64_t K) { return w4a4_q4_0_codes_bytes(rows, K); }
size_t w4a4_act4_expanded_bytes(int64_t rows, int64_t K) { return w4a4_q4_0_expanded_bytes(rows, K); }
size_t w4a4_act8_codes_bytes(int64_t rows, int64_t K) {
  if (!valid_k(K) || rows < 0) return 0;
  return round16(static_cast<size_t>(rows) * static_cast<size_t>(K));
}
size_t w4a4_act8_scales_bytes(int64_t rows, int64_t K) { return w4a4_act4_scales_bytes(rows, K); }
size_t w4a4_act16_values_bytes(int64_t rows, int64_t K) {
  if (!valid_k(K) || rows < 0) return 0;
  return round16(static_cast<size_t>(rows) * static_cast<size_t>(K) * 2);
}
size_t w4a4_act4_scales_bytes(int64_t rows, int64_t K) {
  if (!valid_k(K) || rows < 0) return 0;
  return round16(static_cast<size_t>(rows) * static_cast<size_t>(K / 32) * 4);
}

w4a4_status h32_q4_0_pack_weights(const void* w, int w_dtype, int64_t N, int64_t K, int64_t ldw, int rotate,
                                  w4a4_q4_0* out, w4a4_stream_t stream) {
  const char* fn = "h32_q4_0_pack_weights";
  if (!out) return fail(W4A4_ERR_INVALID_ARG, "%s: out is NULL", fn);
  w4a4_status s = check_k_rows(N, K, fn);
  if (s != W4A4_OK) return s;
  if (w_dtype != W4A4_DTYPE_BF16 && w_dtype != W4A4_DTYPE_F32)
    return fail(W4A4_ERR_INVALID_ARG, "%s: w_dtype %d is neither bf16 (0) nor f32 (1)", fn, w_dtype);
  if (rotate != 0 && rotate != 1) return fail(W4A4_ERR_INVALID_ARG, "%s: rotate must be 0 or 1", fn);
  if (ldw < K) return fail(W4A4_ERR_INVALID_ARG, "%s: ldw=%lld < K=%lld", fn, (long long)ldw, (long long)K);
  const int64_t esz = (w_dtype == W4A4_DTYPE_BF16) ? 2 : 4;
  if (N > 0 && (!w || !out->codes || !out->scales || !out->sums))
    return fail(W4A4_ERR_INVALID_ARG, "%s: NULL pointer", fn);
  if (!aligned16(w) || !aligned16(out->codes) || !aligned16(out->scales) || !aligned16(out->sums) ||
      (ldw * esz) % 16 != 0)
    return fail(W4A4_ERR_ALIGNMENT, "%s: pointers and rows (ldw * element size) must be 16-byte aligned", fn);
  out->rows = N;
  out->K = K;
  out->tag = W4A4_TAG_Q4_0 | (rotate ? W4A4_TAG_ROTATED : 0u);
  if (N == 0) return ok();
  if (!aligned16(out->expanded)) return fail(W4A4_ERR_ALIGNMENT, "%s: expanded must be 16-byte aligned", fn);
  return cuda_status(w4a4::launch_pack_q4_0(w, w_dtype, N, K, ldw, rotate, out->codes, out->scales, out->sums,
                                            out->expanded,
                                            reinterpret_cast<cudaStream_t>(stream)), fn);
}

w4a4_status h32_q4_0_pack_weights_imatrix(const void* w, int w_dtype, int64_t N, int64_t K, int64_t ldw, int rotate,
                                          const float* imatrix, w4a4_q4_0* out, w4a4_stream_t stream) {
  const char* fn = "h32_q4_0_pack_weights_imatrix";
  if (!out) return fail(W4A4_ERR_INVALID_ARG, "%s: out is NULL", fn);
  w4a4_status s = check_k_rows(N, K, fn);
  if (s != W4A4_OK) return s;
  if (w_dtype != W4A4_DTYPE_BF16 && w_dtype != W4A4_DTYPE_F32)
    return fail(W4A4_ERR_INVALID_ARG, "%s: w_dtype %d is neither bf16 (0) nor f32 (1)", fn, w_dtype);
  if (rotate != 0 && rotate != 1) return fail(W4A4_ERR_INVALID_ARG, "%s: rotate must be 0 or 1", fn);
  if (ldw < K) return fail(W4A4_ERR_INVALID_ARG, "%s: ldw=%lld < K=%lld", fn, (long long)ldw, (long long)K);
  const int64_t esz = (w_dtype == W4A4_DTYPE_BF16) ? 2 : 4;
  if (N > 0 && (!w || !out->codes || !out->scales || !out->sums))
    return fail(W4A4_ERR_INVALID_ARG, "%s: NULL pointer", fn);
  if (!aligned16(w) || !aligned16(out->codes) || !aligned16(out->scales) || !aligned16(out->sums) ||
      !aligned16(imatrix) || (ldw * esz) % 16 != 0)
    return fail(W4A4_ERR_ALIGNMENT, "%s: pointers and rows (ldw * element size) must be 16-byte aligned", fn);
  out->rows = N;
  out->K = K;
  out->tag = W4A4_TAG_Q4_0 | (rotate ? W4A4_TAG_ROTATED : 0u);
  if (N == 0) return ok();
  if (!aligned16(out->expanded)) return fail(W4A4_ERR_ALIGNMENT, "%s: expanded must be 16-byte aligned", fn);
  return cuda_status(w4a4::launch_pack_q4_0_weighted(w, w_dtype, N, K, ldw, rotate, imatrix, out->codes, out->scales,
                                                     out->sums, out->expanded, reinterpret_cast<cudaStream_t>(stream)),
                     fn);
}

w4a4_status q4_0_import(const void* blocks, int64_t N, int64_t K, int rotated, w4a4_q4_0* out,
                        w4a4_stream_t stream) {
  const char* fn = "q4_0_import";
  if (!out) return fail(W4A4_ERR_INVALID_ARG, "%s: out is NULL", fn);
  w4a4_status s = check_k_rows(N, K, fn);
  if (s != W4A4_OK) return s;
  if (rotated != 0 && rotated != 1) return fail(W4A4_ERR_INVALID_ARG, "%s: rotated must be 0 or 1", fn);
  if (N > 0 && (!blocks || !out->codes || !out->scales || !out->sums))
    return fail(W4A4_ERR_INVALID_ARG, "%s: NULL pointer", fn);
  if ((reinterpret_cast<uintptr_t>(blocks) & 1u) != 0 || !aligned16(out->codes) || !aligned16(out->scales) ||
      !aligned16(out->sums))
    return fail(W4A4_ERR_ALIGNMENT, "%s: blocks must be 2-byte aligned, outputs 16-byte aligned", fn);
  out->rows = N;
  out->K = K;
  out->tag = W4A4_TAG_Q4_0 | (rotated ? W4A4_TAG_ROTATED : 0u);
  if (N == 0) return ok();
  if (!aligned16(out->expanded)) return fail(W4A4_ERR_ALIGNMENT, "%s: expanded must be 16-byte aligned", fn);
  return cuda_status(w4a4::launch_import_q4_0(blocks, N, K, out->codes, out->scales, out->sums, out->expanded,
                                              reinterpret_cast<cudaStream_t>(stream)), fn);
}

w4a4_status w4a4_rotate_quantize_act(const float* x, int64_t M, int64_t K, int64_t ldx, int rotate,
                                     w4a4_act4* out, w4a4_stream_t stream) {
  const char* fn = "w4a4_rotate_quantize_act";
  if (!out) return fail(W4A4_ERR_INVALID_ARG, "%s: out is NULL", fn);
  w4a4_status s = check_k_rows(M, K, fn);
  if (s != W4A4_OK) return s;
  if (rotate != 0 && rotate != 1) return fail(W4A4_ERR_INVALID_ARG, "%s: rotate must be 0 or 1", fn);
  if (ldx < K) return fail(W4A4_ERR_INVALID_ARG, "%s: ldx=%lld < K=%lld", fn, (long long)ldx, (long long)K);
  if (M > 0 && (!x || !out->codes || !out->scales)) return fail(W4A4_ERR_INVALID_ARG, "%s: NULL pointer", fn);
  if (!aligned16(x) || !aligned16(out->codes) || !aligned16(out->scales) || !aligned16(out->expanded) ||
      (ldx % 4) != 0)
    return fail(W4A4_ERR_ALIGNMENT, "%s: pointers and rows (ldx * 4 bytes) must be 16-byte aligned", fn);
  out->rows = M;
  out->K = K;
  out->tag = W4A4_TAG_ACT4 | (rotate ? W4A4_TAG_ROTATED : 0u);
  if (M == 0) return ok();
  return cuda_status(w4a4::launch_act_rotate_quantize(x, M, K, ldx, rotate, out->codes, out->scales, out->expanded,
                                                      reinterpret_cast<cudaStream_t>(stream)), fn);
}

size_t w4a4_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || !valid_k(K)) return 0;
  const size_t a = w4a4::gemm_workspace_bytes(M, N, K), b = w4a4::grp_workspace_bytes(M, N, K);
  return a > b ? a : b;
}

w4a4_status w4a4_gemm(const w4a4_q4_0* w, const w4a4_act4* a, float* y, int64_t ldy, void* ws, size_t ws_bytes,
                      w4a4_stream_t stream) {
  const char* fn = "w4a4_gemm";
  w4a4_status s = check_q4_0(w, fn);
  if (s != W4A4_OK) return s;
  if ((s = check_act4(a, fn)) != W4A4_OK) return s;
  if ((s = check_pair(w, a, fn)) != W4A4_OK) return s;
  const int64_t M = a->rows, N = w->rows;
  if (ldy < N) return fail(W4A4_ERR_INVALID_ARG, "%s: ldy=%lld < N=%lld", fn, (long long)ldy, (long long)N);
  if (M == 0 || N == 0) return ok();
  if (!y) return fail(W4A4_ERR_INVALID_ARG, "%s: y is NULL", fn);
  if ((reinterpret_cast<uintptr_t>(y) & 3u) != 0) return fail(W4A4_ERR_ALIGNMENT, "%s: y must be 4-byte aligned", fn);
  if (ws) {
    const size_t need = w4a4_gemm_workspace_bytes(M, N, a->K);
    if (ws_bytes < need)
      return fail(W4A4_ERR_WORKSPACE, "%s: workspace %zu bytes < %zu needed", fn, ws_bytes, need);
    if (!aligned16(ws)) return fail(W4A4_ERR_ALIGNMENT, "%s: ws must be 16-byte aligned", fn);
  }
  // with the expanded activation operand: the super-tile kernel; else the kernel that
  // converts both operands' codes
  if (a->expanded)
    return cuda_status(w4a4::launch_gemm_grp(w->codes, w->scales, w->sums, w->expanded, N, a->expanded, a->scales,
                                             M, a->K, y, ldy, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream)),
                       fn);
  return cuda_status(w4a4::launch_gemm_tc(w->codes, w->scales, w->sums, w->expanded, N, a->codes, a->scales,
                                          M, a->K, y, ldy, nullptr, ws, ws_bytes,
                                          reinterpret_cast<cudaStream_t>(stream)), fn);
}

w4a4_status w4a4_gemm_small_m(const w4a4_q4_0* w, const w4a4_act4* a, float* y, int64_t ldy, w4a4_stream_t stream) {
  const char* fn = "w4a4_gemm_small_m";
  w4a4_status s = check_q4_0(w, fn);
  if (s != W4A4_OK) return s;
  if ((s = check_act4(a, fn)) != W4A4_OK) return s;
  if ((s = check_pair(w, a, fn)) != W4A4_OK) return s;
  const int64_t M = a->rows, N = w->rows;
  if (M > 8) return fail(W4A4_ERR_UNSUPPORTED, "%s: %lld activation rows; this kernel takes 1 to 8", fn, (long long)M);
  if (ldy < N) return fail(W4A4_ERR_INVALID_ARG, "%s: ldy=%lld < N=%lld", fn, (long long)ldy, (long long)N);
  if (M == 0 || N == 0) return ok();
  if (!y) return fail(W4A4_ERR_INVALID_ARG, "%s: y is NULL", fn);
  if ((reinterpret_cast<uintptr_t>(y) & 3u) != 0) return fail(W4A4_ERR_ALIGNMENT, "%s: y must be 4-byte aligned", fn);
  return cuda_status(w4a4::launch_gemm_small_m(w->codes, w->scales, N, a->codes, a->scales, static_cast<int>(M), a->K,
                                               y, ldy, reinterpret_cast<cudaStream_t>(stream)), fn);
}

w4a4_status w4a4_gemm_partials(const w4a4_q4_0* w, const w4a4_act4* a, int32_t* P, w4a4_stream_t stream) {
  const char* fn = "w4a4_gemm_partials";
  w4a4_status s = check_q4_0(w, fn);
  if (s != W4A4_OK) return s;
  if ((s = check_act4(a, fn)) != W4A4_OK) return s;
  if ((s = check_pair(w, a, fn)) != W4A4_OK) return s;
  if (a->rows == 0 || w->rows == 0) return ok();
  if (!P) return fail(W4A4_ERR_INVALID_ARG, "%s: P is NULL", fn);
  if (!aligned16(P)) return fail(W4A4_ERR_ALIGNMENT, "%s: P must be 16-byte aligned", fn);
  return cuda_status(w4a4::launch_gemm_tc(w->codes, w->scales, w->sums, nullptr, w->rows, a->codes, a->scales,
                                          a->rows, a->K, nullptr, 0, P, nullptr, 0,
                                          reinterpret_cast<cudaStream_t>(stream)), fn);
}

w4a4_status w4a8_rotate_quantize_act(const float* x, int64_t M, int64_t K, int64_t ldx, int rotate,
                                     w4a4_act8* out, w4a4_stream_t stream) {
  const char* fn = "w4a8_rotate_quantize_act";
  if (!out) return fail(W4A4_ERR_INVALID_ARG, "%s: out is NULL", fn);
  w4a4_status s = check_k_rows(M, K, fn);
  if (s != W4A4_OK) return s;
  if (rotate != 0 && rotate != 1) return fail(W4A4_ERR_INVALID_ARG, "%s: rotate must be 0 or 1", fn);
  if (ldx < K) return fail(W4A4_ERR_INVALID_ARG, "%s: ldx=%lld < K=%lld", fn, (long long)ldx, (long long)K);
  if (M > 0 && (!x || !out->codes || !out->scales)) return fail(W4A4_ERR_INVALID_ARG, "%s: NULL pointer", fn);
  if (!aligned16(x) || !aligned16(out->codes) || !aligned16(out->scales) || (ldx % 4) != 0)
    return fail(W4A4_ERR_ALIGNMENT, "%s: pointers and rows (ldx * 4 bytes) must be 16-byte aligned", fn);
  out->rows = M;
  out->K = K;
  out->tag = W4A4_TAG_ACT8 | (rotate ? W4A4_TAG_ROTATED : 0u);
  if (M == 0) return ok();
  return cuda_status(w4a4::launch_act_rotate_quantize8(x, M, K, ldx, rotate, out->codes, out->scales,
                                                       reinterpret_cast<cudaStream_t>(stream)), fn);
}

size_t w4a8_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || !valid_k(K)) return 0;
  return w4a4::gemm_w4a8_workspace_bytes(M, N, K);
}

w4a4_status w4a8_gemm(const w4a4_q4_0* w, const w4a4_act8* a, float* y, int64_t ldy, void* ws, size_t ws_bytes,
                      w4a4_stream_t stream) {
  const char* fn = "w4a8_gemm";
  w4a4_status s = check_q4_0(w, fn);
  if (s != W4A4_OK) return s;
  if ((s = check_act8(a, fn)) != W4A4_OK) return s;
  if ((s = check_pair(w, a, fn)) != W4A4_OK) return s;
  const int64_t M = a->rows, N = w->rows;
  if (ldy < N) return fail(W4A4_ERR_INVALID_ARG, "%s: ldy=%lld < N=%lld", fn, (long long)ldy, (long long)N);
  if (M == 0 || N == 0) return ok();
  if (!y) return fail(W4A4_ERR_INVALID_ARG, "%s: y is NULL", fn);
  if ((reinterpret_cast<uintptr_t>(y) & 3u) != 0) return fail(W4A4_ERR_ALIGNMENT, "%s: y must be 4-byte aligned", fn);
  if (ws) {
    const size_t need = w4a4::gemm_w4a8_workspace_bytes(M, N, a->K);
    if (ws_bytes < need)
      return fail(W4A4_ERR_WORKSPACE, "%s: workspace %zu bytes < %zu needed", fn, ws_bytes, need);
    if (!aligned16(ws)) return fail(W4A4_ERR_ALIGNMENT, "%s: ws must be 16-byte aligned", fn);
  }
  return cuda_status(w4a4::launch_gemm_w4a8(w->codes, w->scales, w->sums, N, a->codes, a->scales, M, a->K, y, ldy,
                                            nullptr, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream)), fn);
}

w4a4_status w4a16_rotate_act(const float* x, int64_t M, int64_t K, int64_t ldx, int rotate, w4a4_act16* out,
                             w4a4_stream_t stream) {
  const char* fn = "w4a16_rotate_act";
  if (!out) return fail(W4A4_ERR_INVALID_ARG, "%s: out is NULL", fn);
  w4a4_status s = check_k_rows(M, K, fn);
  if (s != W4A4_OK) return s;
  if (rotate != 0 && rotate != 1) return fail(W4A4_ERR_INVALID_ARG, "%s: rotate must be 0 or 1", fn);
  if (ldx < K) return fail(W4A4_ERR_INVALID_ARG, "%s: ldx=%lld < K=%lld", fn, (long long)ldx, (long long)K);
  if (M > 0 && (!x || !out->values)) return fail(W4A4_ERR_INVALID_ARG, "%s: NULL pointer", fn);
  if (!aligned16(x) || !aligned16(out->values) || (ldx % 4) != 0)
    return fail(W4A4_ERR_ALIGNMENT, "%s: pointers and rows (ldx * 4 bytes) must be 16-byte aligned", fn);
  out->rows = M;
  out->K = K;
  out->tag = W4A4_TAG_ACT16 | (rotate ? W4A4_TAG_ROTATED : 0u);
  if (M == 0) return ok();
  return cuda_status(w4a4::launch_act_rotate_bf16(x, M, K, ldx, rotate, out->values,
                                                  reinterpret_cast<cudaStream_t>(stream)), fn);
}

size_t w4a16_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || !valid_k(K)) return 0;
  return w4a4::gemm_w4a8_workspace_bytes(M, N, K);
}

w4a4_status w4a16_gemm(const w4a4_q4_0* w, const w4a4_act16* a, float* y, int64_t ldy, void* ws, size_t ws_bytes,
                       w4a4_stream_t stream) {
  const char* fn = "w4a16_gemm";
  w4a4_status s = check_q4_0(w, fn);
  if (s != W4A4_OK) return s;
  if ((s = check_act16(a, fn)) != W4A4_OK) return s;
  if ((s = check_pair(w, a, fn)) != W4A4_OK) return s;
  const int64_t M = a->rows, N = w->rows;
  if (ldy < N) return fail(W4A4_ERR_INVALID_ARG, "%s: ldy=%lld < N=%lld", fn, (long long)ldy, (long long)N);
  if (M == 0 || N == 0) return ok();
  if (!y) return fail(W4A4_ERR_INVALID_ARG, "%s: y is NULL", fn);
  if ((reinterpret_cast<uintptr_t>(y) & 3u) != 0) return fail(W4A4_ERR_ALIGNMENT, "%s: y must be 4-byte aligned", fn);
  if (ws) {
    const size_t need = w4a4::gemm_w4a8_workspace_bytes(M, N, a->K);
    if (ws_bytes < need)
      return fail(W4A4_ERR_WORKSPACE, "%s: workspace %zu bytes < %zu needed", fn, ws_bytes, need);
    if (!aligned16(ws)) return fail(W4A4_ERR_ALIGNMENT, "%s: ws must be 16-byte aligned", fn);
  }
  return cuda_status(w4a4::launch_gemm_w4a16(w->codes, w->scales, w->sums, N, a->values, M, a->K, y, ldy, ws,
                                             ws_bytes, reinterpret_cast<cudaStream_t>(stream)), fn);
}

w4a4_status w4a8_gemm_partials(const w4a4_q4_0* w, const w4a4_act8* a, int32_t* P, w4a4_stream_t stream) {
  const char* fn = "w4a8_gemm_partials";
  w4a4_status s = check_q4_0(w, fn);
  if (s != W4A4_OK) return s;
  if ((s = check_act8(a, fn)) != W4A4_OK) return s;
  if ((s = check_pair(w, a, fn)) != W4A4_OK) return s;
  if (a->rows == 0 || w->rows == 0) return ok();
  if (!P) return fail(W4A4_ERR_INVALID_ARG, "%s: P is NULL", fn);
  if (!aligned16(P)) return fail(W4A4_ERR_ALIGNMENT, "%s: P must be 16-byte aligned", fn);
  return cuda_status(w4a4::launch_gemm_w4a8(w->codes, w->scales, w->sums, w->rows, a->codes, a->scales, a->rows, a->K,
                                            nullptr, 0, P, nullptr, 0, reinterpret_cast<cudaStream_t>(stream)), fn);
}

size_t w4a4_gemm_id_workspace_bytes(int64_t M, int top_k, int E, int64_t K) {
  if (M < 0 || top_k <= 0 || E <= 0 || !valid_k(K)) return 0;
  return w4a4::routing_layout(M * top_k, E, K).total;
}

w4a4_status w4a4_gemm_id(const w4a4_q4_0* experts, int E, int64_t N, const w4a4_act4* a, const int32_t* ids,
                         int64_t M, int top_k, int act_per_slot, float* y, void* ws, size_t ws_bytes,
                         w4a4_stream_t stream) {
  const char* fn = "w4a4_gemm_id";
  w4a4_status s = check_q4_0(experts, fn);
  if (s != W4A4_OK) return s;
  if ((s = check_act4(a, fn)) != W4A4_OK) return s;
  if ((s = check_pair(experts, a, fn)) != W4A4_OK) return s;
  if (E < 1 || E > 4096) return fail(W4A4_ERR_INVALID_ARG, "%s: E=%d outside 1..4096", fn, E);
  if (top_k < 1 || top_k > E) return fail(W4A4_ERR_INVALID_ARG, "%s: top_k=%d outside 1..E", fn, top_k);
  if (N < 1) return fail(W4A4_ERR_INVALID_ARG, "%s: N=%lld must be positive", fn, (long long)N);
  if (M < 0 || M * top_k > (int64_t(1) << 31) - 1) return fail(W4A4_ERR_INVALID_ARG, "%s: bad M", fn);
  if (act_per_slot != 0 && act_per_slot != 1) return fail(W4A4_ERR_INVALID_ARG, "%s: act_per_slot must be 0 or 1", fn);
  if (experts->rows != static_cast<int64_t>(E) * N)
    return fail(W4A4_ERR_MISMATCH, "%s: expert weights have %lld rows, expected E*N = %lld", fn,
                (long long)experts->rows, (long long)(static_cast<int64_t>(E) * N));
  const int64_t want_rows = act_per_slot ? M * top_k : M;
  if (a->rows != want_rows)
    return fail(W4A4_ERR_MISMATCH, "%s: activations have %lld rows, expected %lld", fn, (long long)a->rows,
                (long long)want_rows);
  if (M == 0) return ok();
  if (!ids || !y || !ws) return fail(W4A4_ERR_INVALID_ARG, "%s: NULL pointer", fn);
  const size_t need = w4a4_gemm_id_workspace_bytes(M, top_k, E, a->K);
  if (ws_bytes < need) return fail(W4A4_ERR_WORKSPACE, "%s: workspace %zu bytes < %zu needed", fn, ws_bytes, need);
  if (!aligned16(ws) || (reinterpret_cast<uintptr_t>(y) & 3u) != 0)
    return fail(W4A4_ERR_ALIGNMENT, "%s: ws must be 16-byte aligned and y 4-byte aligned", fn);
  const w4a4::Routing r = w4a4::routing_in(ws, M * top_k, E, a->K);
  return cuda_status(w4a4::launch_gemm_id(experts->codes, experts->scales, experts->sums, E, N, a->codes, a->scales, a->K, ids, M,
                                          top_k, act_per_slot, y, r, reinterpret_cast<cudaStream_t>(stream)), fn);
}

w4a4_status w4a4_gemm_id_status(const void* ws, w4a4_stream_t stream) {
  const char* fn = "w4a4_gemm_id_status";
  if (!ws) return fail(W4A4_ERR_INVALID_ARG, "%s: ws is NULL", fn);
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_status(e, fn);
  int32_t flag = 0;  // the routing flag is the first word of the workspace
  e = cudaMemcpy(&flag, ws, sizeof(flag), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_status(e, fn);
  if (flag != 0) return fail(W4A4_ERR_DEVICE_FLAG, "%s: an expert id was outside [0, E); its rows were zeroed", fn);
  return ok();
}

static_assert(W4A4_GEMM_ID_STATIC_SCRATCH_BYTES == w4a4::kIdStaticScratchBytes, "scratch size mismatch");

w4a4_status w4a4_gemm_id_static(const w4a4_q4_0* experts, int E, int64_t N, const w4a4_act4* a, const int32_t* ids,
                                int64_t M, int top_k, int act_per_slot, float* y, w4a4_stream_t stream) {
  const char* fn = "w4a4_gemm_id_static";
  w4a4_status s = check_q4_0(experts, fn);
  if (s != W4A4_OK) return s;
  if ((s = check_act4(a, fn)) != W4A4_OK) return s;
  if ((s = check_pair(experts, a, fn)) != W4A4_OK) return s;
  if (E < 1 || E > 4096) return fail(W4A4_ERR_INVALID_ARG, "%s: E=%d outside 1..4096", fn, E);
  if (top_k < 1 || top_k > E) return fail(W4A4_ERR_INVALID_ARG, "%s: top_k=%d outside 1..E", fn, top_k);
  if (N < 1) return fail(W4A4_ERR_INVALID_ARG, "%s: N=%lld must be positive", fn, (long long)N);
  if (M < 0 || M * top_k > (int64_t(1) << 31) - 1) return fail(W4A4_ERR_INVALID_ARG, "%s: bad M", fn);
  if (act_per_slot != 0 && act_per_slot != 1) return fail(W4A4_ERR_INVALID_ARG, "%s: act_per_slot must be 0 or 1", fn);
  if (experts->rows != static_cast<int64_t>(E) * N)
    return fail(W4A4_ERR_MISMATCH, "%s: expert weights have %lld rows, expected E*N = %lld", fn,
                (long long)experts->rows, (long long)(static_cast<int64_t>(E) * N));
  const int64_t want_rows = act_per_slot ? M * top_k : M;
  if (a->rows != want_rows)
    return fail(W4A4_ERR_MISMATCH, "%s: activations have %lld rows, expected %lld", fn, (long long)a->rows,
                (long long)want_rows);
  if (M == 0) return ok();
  if (!ids || !y) return fail(W4A4_ERR_INVALID_ARG, "%s: NULL pointer", fn);
  const size_t need = w4a4_gemm_id_workspace_bytes(M, top_k, E, a->K);
  if (need > W4A4_GEMM_ID_STATIC_SCRATCH_BYTES)
    return fail(W4A4_ERR_WORKSPACE,
                "%s: this problem needs %zu bytes of routing scratch, more than the fixed %zu; "
                "call w4a4_gemm_id with a workspace instead",
                fn, need, static_cast<size_t>(W4A4_GEMM_ID_STATIC_SCRATCH_BYTES));
  if ((reinterpret_cast<uintptr_t>(y) & 3u) != 0) return fail(W4A4_ERR_ALIGNMENT, "%s: y must be 4-byte aligned", fn);
  void* ws = nullptr;
  cudaError_t e = w4a4::id_static_scratch(&ws);
  if (e != cudaSuccess) return cuda_status(e, fn);
  const w4a4::Routing r = w4a4::routing_in(ws, M * top_k, E, a->K);
  return cuda_status(w4a4::launch_gemm_id(experts->codes, experts->scales, experts->sums, E, N, a->codes, a->scales,
                                          a->K, ids, M, top_k, act_per_slot, y, r,
                                          reinterpret_cast<cudaStream_t>(stream)),
                     fn);
}

w4a4_status w4a4_check(w4a4_stream_t stream) {
  const char* fn = "w4a4_check";
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_status(e, fn);
  int flag = 0;
  e = w4a4::read_and_clear_device_error(&flag);
  if (e != cudaSuccess) return cuda_status(e, fn);
  if (flag != 0)
    return fail(W4A4_ERR_TIMEOUT, "%s: a bounded wait inside a GEMM kernel gave up; its output is incomplete", fn);
  return ok();
}

void w4a4_debug_set_wait_limit(uint64_t wait_ns, uint64_t producer_delay_ns) {
  w4a4::grp_set_wait_limit(wait_ns, producer_delay_ns);
}

const char* w4a4_last_error(void) { return g_err; }

const char* w4a4_status_name(w4a4_status s) {
  switch (s) {
    case W4A4_OK: return "W4A4_OK";
    case W4A4_ERR_INVALID_ARG: return "W4A4_ERR_INVALID_ARG";
    case W4A4_ERR_ALIGNMENT: return "W4A4_ERR_ALIGNMENT";
    case W4A4_ERR_MISMATCH: return "W4A4_ERR_MISMATCH";
    case W4A4_ERR_UNSUPPORTED: return "W4A4_ERR_UNSUPPORTED";
    case W4A4_ERR_CUDA: return "W4A4_ERR_CUDA";
    case W4A4_ERR_DEVICE_FLAG: return "W4A4_ERR_DEVICE_FLAG";
    case W4A4_ERR_WORKSPACE: return "W4A4_ERR_WORKSPACE";
    case W4A4_ERR_TIMEOUT: return "W4A4_ERR_TIMEOUT";
  }
  return "W4A4_ERR_UNKNOWN";
}

int w4a4_abi_version(void) { return 200; }

}  // extern "C"
