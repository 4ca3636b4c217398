// Block-scaled W4A4 product for small token batches (M <= 8): verification
// batches of a drafter (engine docs "The lean option: ROCmFP4, ROCmI4 and
// Hadamard Q4_0", a row-tiled Q4_0 kernel for 8-column verification batches:
// one warp computes 4 weight rows, each weight is unpacked once for all columns,
// and the output is bit for bit that of the general kernel).
//
// With M <= 8 the product is a weight stream: the tensor-core tile (128 weight
// rows x 32+ token columns) would leave most of its MMA and fold idle.  Here a
// CTA owns 32 weight rows and walks K in chunks of 64 blocks:
//   * the chunk's weight codes and scales (32 rows x 1 KB + 4 KB) are copied
//     into shared memory with cp.async, one chunk ahead of the one computed, so
//     every SM keeps tens of KB of weight reads in flight;
//   * the chunk's activation codes are widened to int8 in shared memory, with
//     each block's code sum S_a and scale d_a;
//   * warp w computes rows 4w .. 4w+3, lane l the output (row 4w + l / 8, token
//     l % 8); per block P = sum_j (q - 8) a_j = dp4a(q, a) - 8 S_a exactly, with
//     the unsigned codes q (0..15 are the same as signed bytes);
//   * the fold is the general kernel's, in the same order: t = round(d_w P),
//     acc = fma(t, d_a, acc) over the blocks in order, so for the general
//     kernel's whole-tile schedule the results agree bit for bit.
// Shared-memory rows are padded so that the 8 token rows (and the 4 weight rows
// a warp reads at once) fall in distinct banks.
#include "w4a4_kernels.cuh"

namespace w4a4 {

namespace {

#ifndef W4A4_SM_WARPS
#define W4A4_SM_WARPS 4
#endif
#ifndef W4A4_SM_CHUNK
#define W4A4_SM_CHUNK 64
#endif
#ifndef W4A4_SM_UNROLL
#define W4A4_SM_UNROLL 8
#endif
constexpr int kSmWarps = W4A4_SM_WARPS;
constexpr int kSmUnroll = W4A4_SM_UNROLL;
constexpr int kSmRows = 4 * kSmWarps;  // weight rows per CTA (4 per warp)
constexpr int kSmMaxM = 8;
constexpr int kSmChunk = W4A4_SM_CHUNK;  // blocks per chunk (16 code bytes each per weight row)
constexpr int kWRow = kSmChunk * 16 + 16;      // weight code bytes per row, padded by 16
constexpr int kARow = kSmChunk * 8 + 4;        // int8 activation words per row, padded by 4
constexpr int kSRow = kSmChunk + 4;            // fp16 weight scales per row, padded (8-byte rows, distinct banks)

struct SmallMSmem {
  uint8_t w[2][kSmRows][kWRow];           // weight codes of two chunks
  uint16_t ws[2][kSmRows][kSRow];         // their fp16 scales
  uint32_t a8[kSmMaxM][kARow];            // int8 activation codes, 4 per word, element order
  float da[kSmChunk][kSmMaxM];            // d_a, block-major
  int32_t sa[kSmChunk][kSmMaxM];          // 8 S_a, block-major
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async8(void* smem, const void* gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Four 4-bit two's complement nibbles (the low nibble of each byte of v) as
// four signed bytes: bit 3 of each byte, times 30 (0x08 * 30 = 0xF0), fills its
// high nibble; no product crosses a byte.
__device__ __forceinline__ uint32_t s4x4_to_s8x4(uint32_t v) {
  const uint32_t x = v & 0x0F0F0F0Fu;
  return x | ((x & 0x08080808u) * 30u);
}

// Copy chunk c's weight codes and scales of this CTA's rows (rows past N and
// blocks past B are not copied; they are never read).
__device__ __forceinline__ void load_weight_chunk(SmallMSmem& S, int buf, const uint8_t* w_codes,
                                                  const uint16_t* w_scales, int64_t n0, int64_t N, int64_t K,
                                                  int64_t b0, int nb) {
  const int64_t B = K / 32;
  // codes: 32 rows x nb 16-byte pieces
  for (int idx = threadIdx.x; idx < kSmRows * nb; idx += blockDim.x) {
    const int r = idx / nb, bb = idx - r * nb;
    if (n0 + r < N) cp_async16(&S.w[buf][r][bb * 16], w_codes + (n0 + r) * (K / 2) + (b0 + bb) * 16);
  }
  // scales: 4 fp16 (8 bytes) per piece when aligned, else one by one
  if ((B & 3) == 0 && (b0 & 3) == 0 && (nb & 3) == 0) {
    for (int idx = threadIdx.x; idx < kSmRows * (nb / 4); idx += blockDim.x) {
      const int r = idx / (nb / 4), q = idx - r * (nb / 4);
      if (n0 + r < N) cp_async8(&S.ws[buf][r][4 * q], w_scales + (n0 + r) * B + b0 + 4 * q);
    }
  } else {
    for (int idx = threadIdx.x; idx < kSmRows * nb; idx += blockDim.x) {
      const int r = idx / nb, bb = idx - r * nb;
      if (n0 + r < N) S.ws[buf][r][bb] = w_scales[(n0 + r) * B + b0 + bb];
    }
  }
}

__global__ void __launch_bounds__(32 * kSmWarps) w4a4_small_m_kernel(
    const uint8_t* __restrict__ w_codes, const uint16_t* __restrict__ w_scales, int64_t N,
    const uint8_t* __restrict__ a_codes, const float* __restrict__ a_scales, int M, int64_t K,
    float* __restrict__ y, int64_t ldy) {
  extern __shared__ __align__(16) uint8_t sm_raw[];
  SmallMSmem& S = *reinterpret_cast<SmallMSmem*>(sm_raw);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kSmRows;
  const int r = warp * 4 + (lane >> 3);  // this lane's weight row within the CTA
  const int m = lane & 7;
  const bool live = n0 + r < N && m < M;
  const int64_t B = K / 32;
  const int nchunks = static_cast<int>((B + kSmChunk - 1) / kSmChunk);
  float acc = 0.f;

  load_weight_chunk(S, 0, w_codes, w_scales, n0, N, K, 0, static_cast<int>(B < kSmChunk ? B : kSmChunk));
  cp_async_commit();
  for (int c = 0; c < nchunks; ++c) {
    const int64_t b0 = static_cast<int64_t>(c) * kSmChunk;
    const int nb = static_cast<int>(B - b0 < kSmChunk ? B - b0 : kSmChunk);
    const int buf = c & 1;
    // the next chunk's weights stream in while this one is computed
    if (c + 1 < nchunks) {
      const int64_t b1 = b0 + kSmChunk;
      load_weight_chunk(S, buf ^ 1, w_codes, w_scales, n0, N, K, b1,
                        static_cast<int>(B - b1 < kSmChunk ? B - b1 : kSmChunk));
    }
    cp_async_commit();
    // stage this chunk's activations: one thread per (row, block)
    for (int idx = threadIdx.x; idx < M * nb; idx += blockDim.x) {
      const int mm = idx / nb, bb = idx - mm * nb;
      const uint4 cw = *reinterpret_cast<const uint4*>(a_codes + mm * (K / 2) + (b0 + bb) * 16);
      // word t: elements 4t..4t+3 in the low nibbles, 16+4t..16+4t+3 in the high ones
      const uint4 lo = make_uint4(s4x4_to_s8x4(cw.x), s4x4_to_s8x4(cw.y), s4x4_to_s8x4(cw.z), s4x4_to_s8x4(cw.w));
      const uint4 hi = make_uint4(s4x4_to_s8x4(cw.x >> 4), s4x4_to_s8x4(cw.y >> 4), s4x4_to_s8x4(cw.z >> 4),
                                  s4x4_to_s8x4(cw.w >> 4));
      int32_t sum = 0;  // S_a: every signed byte times one
      sum = __dp4a(static_cast<int>(lo.x), 0x01010101, sum);
      sum = __dp4a(static_cast<int>(lo.y), 0x01010101, sum);
      sum = __dp4a(static_cast<int>(lo.z), 0x01010101, sum);
      sum = __dp4a(static_cast<int>(lo.w), 0x01010101, sum);
      sum = __dp4a(static_cast<int>(hi.x), 0x01010101, sum);
      sum = __dp4a(static_cast<int>(hi.y), 0x01010101, sum);
      sum = __dp4a(static_cast<int>(hi.z), 0x01010101, sum);
      sum = __dp4a(static_cast<int>(hi.w), 0x01010101, sum);
      *reinterpret_cast<uint4*>(&S.a8[mm][bb * 8]) = lo;
      *reinterpret_cast<uint4*>(&S.a8[mm][bb * 8 + 4]) = hi;
      S.sa[bb][mm] = 8 * sum;
      S.da[bb][mm] = a_scales[mm * B + b0 + bb];
    }
    cp_async_wait<1>();  // this chunk's weights have landed (the next chunk's may be in flight)
    __syncthreads();
    if (live) {
      const uint8_t* wr = &S.w[buf][r][0];
      const uint16_t* wsr = &S.ws[buf][r][0];
      const uint32_t* ar = &S.a8[m][0];
      // t_b = round(d_w P_b) for a group of blocks is independent work; only the
      // folds into acc are chained, and they stay in block order
      auto t_of = [&](int bb) -> float {
        const uint4 cw = *reinterpret_cast<const uint4*>(wr + bb * 16);
        const float dw = __half2float(__ushort_as_half(wsr[bb]));
        const uint4 a0 = *reinterpret_cast<const uint4*>(ar + bb * 8);
        const uint4 a1 = *reinterpret_cast<const uint4*>(ar + bb * 8 + 4);
        const uint32_t wv[4] = {cw.x, cw.y, cw.z, cw.w};
        const uint32_t lo[4] = {a0.x, a0.y, a0.z, a0.w}, hi[4] = {a1.x, a1.y, a1.z, a1.w};
        int32_t pl = 0, ph = 0;  // sum_j q_j a_j with the unsigned codes q, in two independent halves
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          pl = __dp4a(static_cast<int>(wv[t] & 0x0F0F0F0Fu), static_cast<int>(lo[t]), pl);
          ph = __dp4a(static_cast<int>((wv[t] >> 4) & 0x0F0F0F0Fu), static_cast<int>(hi[t]), ph);
        }
        return __fmul_rn(dw, static_cast<float>(pl + ph - S.sa[bb][m]));
      };
      int bb = 0;
      for (; bb + kSmUnroll <= nb; bb += kSmUnroll) {
        float tv[kSmUnroll];
#pragma unroll
        for (int u = 0; u < kSmUnroll; ++u) tv[u] = t_of(bb + u);
#pragma unroll
        for (int u = 0; u < kSmUnroll; ++u) acc = __fmaf_rn(tv[u], S.da[bb + u][m], acc);
      }
      for (; bb < nb; ++bb) acc = __fmaf_rn(t_of(bb), S.da[bb][m], acc);
    }
    __syncthreads();  // the chunk's buffers are free for the loads issued next
  }
  cp_async_wait<0>();
  if (live) y[static_cast<int64_t>(m) * ldy + n0 + r] = acc;
}

}  // namespace

cudaError_t launch_gemm_small_m(const uint8_t* w_codes, const uint16_t* w_scales, int64_t N, const uint8_t* a_codes,
                                const float* a_scales, int M, int64_t K, float* y, int64_t ldy, cudaStream_t stream) {
  if (M < 1 || M > kSmMaxM) return cudaErrorInvalidValue;
  const int64_t grid = (N + kSmRows - 1) / kSmRows;
  if (grid < 1) return cudaSuccess;
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(w4a4_small_m_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(sizeof(SmallMSmem)));
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  w4a4_small_m_kernel<<<static_cast<unsigned>(grid), 32 * kSmWarps, sizeof(SmallMSmem), stream>>>(
      w_codes, w_scales, N, a_codes, a_scales, M, K, y, ldy);
  return cudaGetLastError();
}

}  // namespace w4a4
