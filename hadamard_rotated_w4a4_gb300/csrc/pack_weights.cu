// Weight rotation + Q4_0 packing, and the import of existing Q4_0 blocks.
//
// Engine docs "The lean option: ROCmFP4, ROCmI4 and Hadamard Q4_0", section
// "Hadamard-rotated Q4_0: W4A4 prompt processing": the weights are rotated once
// per 32-element block along K with the same 32-point Walsh-Hadamard transform
// as the activations, then stored as plain Q4_0 (a code q stands for q - 8) and
// read bit for bit; section "MoE: W4A4 on the experts": one scale per 32 values.
//
// Same lane layout as the activation kernel: eight lanes per block, four
// values per lane, butterfly stages h = 1, 2 in registers and h = 4, 8, 16 by
// shuffles.  Runs once per model, so it is written for clarity over speed.
#include "w4a4_kernels.cuh"

namespace w4a4 {

namespace {

__device__ __forceinline__ float4 load4(const void* w, int w_dtype, int64_t off) {
  if (w_dtype == 0) {  // bf16: widen exactly
    const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(w) + off);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xFFFF0000u));
  }
  return *reinterpret_cast<const float4*>(static_cast<const float*>(w) + off);
}

__device__ __forceinline__ float bfly(float v, int bit, bool upper) {
  const float o = __shfl_xor_sync(0xFFFFFFFFu, v, bit);
  return upper ? __fsub_rn(o, v) : __fadd_rn(v, o);
}

// Keep the candidate with the larger magnitude; on equal magnitude the lower index.
__device__ __forceinline__ void keep_larger(float& mval, float& mabs, int& midx, float ov, float oa, int oi) {
  if (oa > mabs || (oa == mabs && oi < midx)) {
    mval = ov;
    mabs = oa;
    midx = oi;
  }
}

// This lane's four values (elements 4t .. 4t+3) of block (n, b), rotated when
// `rotate`: butterfly stages h = 1, 2 in registers, h = 4, 8, 16 by shuffles,
// then one multiply by fl32(1/sqrt 32).
__device__ __forceinline__ void load_block4(const void* w, int w_dtype, int64_t n, int64_t b, int64_t ldw, int t,
                                            bool ok, int rotate, float (&v)[4]) {
  v[0] = v[1] = v[2] = v[3] = 0.f;
  if (ok) {
    const float4 f = load4(w, w_dtype, n * ldw + b * 32 + 4 * t);
    v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
  }
  if (rotate) {
    float a0 = __fadd_rn(v[0], v[1]), a1 = __fsub_rn(v[0], v[1]);
    float a2 = __fadd_rn(v[2], v[3]), a3 = __fsub_rn(v[2], v[3]);
    v[0] = __fadd_rn(a0, a2);
    v[2] = __fsub_rn(a0, a2);
    v[1] = __fadd_rn(a1, a3);
    v[3] = __fsub_rn(a1, a3);
#pragma unroll
    for (int s = 0; s < 3; ++s) {
      const int bit = 1 << s;
      const bool up = (t & bit) != 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = bfly(v[j], bit, up);
    }
    const float c = c_h32();
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = __fmul_rn(v[j], c);
  }
}

// The block's signed value of largest magnitude, lowest index on ties (same in all 8 lanes).
__device__ __forceinline__ float block_signed_max(const float (&v)[4], int t) {
  float mval = v[0], mabs = fabsf(v[0]);
  int midx = 4 * t;
#pragma unroll
  for (int j = 1; j < 4; ++j) {
    const float aj = fabsf(v[j]);
    if (aj > mabs) {
      mabs = aj;
      mval = v[j];
      midx = 4 * t + j;
    }
  }
#pragma unroll
  for (int s = 0; s < 3; ++s) {
    const int bit = 1 << s;
    const float ov = __shfl_xor_sync(0xFFFFFFFFu, mval, bit);
    const float oa = __shfl_xor_sync(0xFFFFFFFFu, mabs, bit);
    const int oi = __shfl_xor_sync(0xFFFFFFFFu, midx, bit);
    keep_larger(mval, mabs, midx, ov, oa, oi);
  }
  return mval;
}

// Code of value x for the reciprocal scale inv: clamp(round_half_away(x * inv) + 8, 0, 15).
__device__ __forceinline__ int q4_code(float x, float inv) {
  const float r = round_half_away(__fmul_rn(x, inv));
  return static_cast<int>(fminf(fmaxf(__fadd_rn(r, 8.0f), 0.0f), 15.0f));
}

// The expanded operand byte of a code: q - 8 as an fp8 e4m3 subnormal
// ((q - 8) * 2^-9), sign and magnitude: q - 8 >= 0 -> q - 8, else 0x80 | (8 - q).
__device__ __forceinline__ uint32_t e4m3_of_code(int q) {
  return static_cast<uint32_t>(q >= 8 ? q - 8 : 0x80 | (8 - q));
}

// Codes of the block for the reciprocal scale inv; stores the 16 code bytes, the
// fp16 scale bits, the code sum sum_j (q_j - 8) and, when `expanded` is given,
// the 32 operand bytes of the block in element order.
__device__ __forceinline__ void store_block(const float (&v)[4], float inv, uint16_t dbits, int t, bool ok, int64_t n,
                                            int64_t b, int64_t K, uint8_t* __restrict__ codes,
                                            uint16_t* __restrict__ scales, int16_t* __restrict__ sums,
                                            uint8_t* __restrict__ expanded) {
  const int64_t B = K / 32;
  uint32_t lo = 0, ex = 0;
  int qsum = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int q = q4_code(v[j], inv);
    lo |= static_cast<uint32_t>(q) << (8 * j);
    ex |= e4m3_of_code(q) << (8 * j);
    qsum += q - 8;
  }
  qsum += __shfl_xor_sync(0xFFFFFFFFu, qsum, 1);
  qsum += __shfl_xor_sync(0xFFFFFFFFu, qsum, 2);
  qsum += __shfl_xor_sync(0xFFFFFFFFu, qsum, 4);
  const uint32_t hi = __shfl_down_sync(0xFFFFFFFFu, lo << 4, 4);
  if (ok) {
    if (expanded) reinterpret_cast<uint32_t*>(expanded + n * K + b * 32)[t] = ex;  // elements 4t..4t+3
    if (t < 4) reinterpret_cast<uint32_t*>(codes + n * (K / 2) + b * 16)[t] = lo | hi;
    if (t == 0) {
      scales[n * B + b] = dbits;
      sums[n * B + b] = static_cast<int16_t>(qsum);
    }
  }
}

__global__ void __launch_bounds__(256) pack_q4_0_kernel(const void* __restrict__ w, int w_dtype, int64_t N,
                                                         int64_t K, int64_t ldw, int rotate,
                                                         uint8_t* __restrict__ codes,
                                                         uint16_t* __restrict__ scales,
                                                         int16_t* __restrict__ sums,
                                                         uint8_t* __restrict__ expanded) {
  const int lane = threadIdx.x & 31;
  const int sub = lane >> 3;
  const int t = lane & 7;
  const int64_t B = K / 32;
  const int64_t nblk = N * B;
  const int64_t ngroups = (nblk + 3) / 4;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t g = warp; g < ngroups; g += nwarps) {
    const int64_t idx = g * 4 + sub;
    const bool ok = idx < nblk;
    const int64_t n = ok ? idx / B : 0;
    const int64_t b = ok ? idx - n * B : 0;
    float v[4];
    load_block4(w, w_dtype, n, b, ldw, t, ok, rotate, v);
    // d = m / -8 with m the signed max; the codes use the fp32 d, the stored scale is fp16(d)
    const float d = __fdiv_rn(block_signed_max(v, t), -8.0f);
    const float inv = (d != 0.0f) ? __frcp_rn(d) : 0.0f;
    store_block(v, inv, __half_as_ushort(__float2half_rn(d)), t, ok, n, b, K, codes, scales, sums, expanded);
  }
}

// ---------------------------------------------------------------------------
// Importance-weighted Q4_0 (the converter's imatrix quantisation, section
// "Hadamard-rotated Q4_0: W4A4 prompt processing": the weights are quantised
// with the importance matrix given the change matching the rotation).
//
// Per block, with weights om_j >= 0: the scale d minimising
// sum_j om_j (y_j - d c_j)^2, each c_j the nearest integer to y_j / d in -8..7.
// With s = 1/d the nearest codes change only where some y_j s crosses k + 1/2
// (k = -8..6); between crossings the codes are fixed and the best d is the
// weighted least-squares num / den (num = sum om y c, den = sum om c^2, error
// sum om y^2 - num^2 / den).  Every crossing is tried from both sides (s times
// 1 -+ 2^-18, far above fp32 rounding and below any interval that matters), the
// codes of all 32 values evaluated at that s, and the largest num^2 / den kept.
// The 8 lanes of a block split the crossings (lane t: those of its elements
// 4t..4t+3) and agree on the best by a symmetric shuffle reduction.  When the
// best codes avoid -8, (-d, -c) is an equally good twin and the sign of the
// plain scale m / -8 is kept (a canonical choice for ties).  The stored
// scale is then the best of fp16(m / -8), fp16(d) and fp16(d)'s two fp16
// neighbours by the weighted error under the Q4_0 code rule, first smallest in
// that order.
//
// The rotated importance is diag(Hn diag(imp) Hn^T): every entry of H32 is
// +-1, so it is the block's mean importance, flat across the block.
constexpr float kSideEps = 0x1p-18f;

// Keep (on, od) from lane ot over (bn, bd) from lane bt when its num^2 / den is
// larger, or equal and from a lower lane (den == 0: no candidate).
__device__ __forceinline__ void keep_better(float& bn, float& bd, float& bs, int& bt, float on, float od, float os,
                                            int ot) {
  if (od <= 0.f) return;
  if (bd <= 0.f) {
    bn = on; bd = od; bs = os; bt = ot;
    return;
  }
  const float lhs = __fmul_rn(__fmul_rn(on, on), bd), rhs = __fmul_rn(__fmul_rn(bn, bn), od);
  if (lhs > rhs || (lhs == rhs && ot < bt)) {
    bn = on; bd = od; bs = os; bt = ot;
  }
}

// fp16 neighbour of bits h toward -inf (up = false) or +inf (up = true).
__device__ __forceinline__ uint16_t half_next(uint16_t h, bool up) {
  const bool neg = (h & 0x8000u) != 0;
  if ((h & 0x7FFFu) == 0) return up ? 0x0001u : 0x8001u;  // from +-0
  return static_cast<uint16_t>((up != neg) ? h + 1 : h - 1);
}

__device__ __forceinline__ float sum8(float x) {  // the same total in every lane of the 8
  x = __fadd_rn(x, __shfl_xor_sync(0xFFFFFFFFu, x, 1));
  x = __fadd_rn(x, __shfl_xor_sync(0xFFFFFFFFu, x, 2));
  return __fadd_rn(x, __shfl_xor_sync(0xFFFFFFFFu, x, 4));
}

__global__ void __launch_bounds__(256) pack_q4_0_weighted_kernel(const void* __restrict__ w, int w_dtype, int64_t N,
                                                                  int64_t K, int64_t ldw, int rotate,
                                                                  const float* __restrict__ imp,
                                                                  uint8_t* __restrict__ codes,
                                                                  uint16_t* __restrict__ scales,
                                                                  int16_t* __restrict__ sums,
                                                                  uint8_t* __restrict__ expanded) {
  __shared__ __align__(16) float s_y[8][4][32];
  __shared__ __align__(16) float s_w[8][4][32];
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const int sub = lane >> 3;
  const int t = lane & 7;
  const int64_t B = K / 32;
  const int64_t nblk = N * B;
  const int64_t ngroups = (nblk + 3) / 4;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t g = warp; g < ngroups; g += nwarps) {
    const int64_t idx = g * 4 + sub;
    const bool ok = idx < nblk;
    const int64_t n = ok ? idx / B : 0;
    const int64_t b = ok ? idx - n * B : 0;
    float v[4];
    load_block4(w, w_dtype, n, b, ldw, t, ok, rotate, v);
    // this lane's four importance values: negative or non-finite count as 0
    float om[4] = {1.f, 1.f, 1.f, 1.f};
    if (imp) {
      const float4 f = ok ? *reinterpret_cast<const float4*>(imp + b * 32 + 4 * t) : make_float4(1.f, 1.f, 1.f, 1.f);
      om[0] = f.x; om[1] = f.y; om[2] = f.z; om[3] = f.w;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) om[j] = (om[j] > 0.f && om[j] <= 3.4028235e38f) ? om[j] : 0.f;
    if (rotate) {  // the matching change: the block mean, flat across the block
      const float mean = __fdiv_rn(sum8(__fadd_rn(__fadd_rn(om[0], om[1]), __fadd_rn(om[2], om[3]))), 32.0f);
#pragma unroll
      for (int j = 0; j < 4; ++j) om[j] = mean;
    }
    // all-zero weights count as uniform; a power-of-two rescale (exact) keeps the
    // products in range and leaves every comparison unchanged
    float mx = fmaxf(fmaxf(om[0], om[1]), fmaxf(om[2], om[3]));
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 4));
    if (mx == 0.f) {
#pragma unroll
      for (int j = 0; j < 4; ++j) om[j] = 1.f;
    } else {  // times 2^(126 - exponent field of mx): mx lands in [0.5, 1)
      const int ex = static_cast<int>((__float_as_uint(mx) >> 23) & 0xFFu);
      const float sc = ex == 0 ? 1.0f : __uint_as_float(static_cast<uint32_t>(ex <= 252 ? 253 - ex : 1) << 23);
#pragma unroll
      for (int j = 0; j < 4; ++j) om[j] = __fmul_rn(om[j], sc);
    }
    *reinterpret_cast<float4*>(&s_y[wib][sub][4 * t]) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4*>(&s_w[wib][sub][4 * t]) = make_float4(om[0], om[1], om[2], om[3]);
    __syncwarp();
    float y[32], wt[32], wy[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 a = *reinterpret_cast<const float4*>(&s_y[wib][sub][4 * i]);
      const float4 c = *reinterpret_cast<const float4*>(&s_w[wib][sub][4 * i]);
      y[4 * i] = a.x; y[4 * i + 1] = a.y; y[4 * i + 2] = a.z; y[4 * i + 3] = a.w;
      wt[4 * i] = c.x; wt[4 * i + 1] = c.y; wt[4 * i + 2] = c.z; wt[4 * i + 3] = c.w;
    }
    __syncwarp();  // the stash is read: the next group may overwrite it
#pragma unroll
    for (int i = 0; i < 32; ++i) wy[i] = __fmul_rn(wt[i], y[i]);
    float bn = 0.f, bd = 0.f, bs = 0.f;  // best num, den and the s that gave its codes
    int bt = t;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      if (v[jj] == 0.f) continue;
#pragma unroll 1
      for (int k = -8; k <= 6; ++k) {
        const float base = __fdiv_rn(static_cast<float>(k) + 0.5f, v[jj]);
#pragma unroll
        for (int side = 0; side < 2; ++side) {
          const float sc = __fmul_rn(base, side ? 1.0f + kSideEps : 1.0f - kSideEps);
          float num = 0.f, den = 0.f;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float c = fminf(fmaxf(rintf(__fmul_rn(y[i], sc)), -8.0f), 7.0f);
            num = __fmaf_rn(wy[i], c, num);
            den = __fmaf_rn(__fmul_rn(wt[i], c), c, den);
          }
          keep_better(bn, bd, bs, bt, num, den, sc, t);
        }
      }
    }
#pragma unroll
    for (int s = 0; s < 3; ++s) {
      const int bit = 1 << s;
      const float on = __shfl_xor_sync(0xFFFFFFFFu, bn, bit);
      const float od = __shfl_xor_sync(0xFFFFFFFFu, bd, bit);
      const float os = __shfl_xor_sync(0xFFFFFFFFu, bs, bit);
      const int ot = __shfl_xor_sync(0xFFFFFFFFu, bt, bit);
      keep_better(bn, bd, bs, bt, on, od, os, ot);
    }
    const float dplain = __fdiv_rn(block_signed_max(v, t), -8.0f);
    float dstar = bd > 0.f ? __fdiv_rn(bn, bd) : 0.f;
    bool uses_m8 = false;  // do the best codes use -8 (then no equally good twin)?
#pragma unroll
    for (int i = 0; i < 32; ++i) uses_m8 |= fminf(fmaxf(rintf(__fmul_rn(y[i], bs)), -8.0f), 7.0f) == -8.0f;
    if (!uses_m8 && dstar * dplain < 0.f) dstar = -dstar;
    const uint16_t plain = __half_as_ushort(__float2half_rn(dplain));
    const uint16_t ds = __half_as_ushort(__float2half_rn(dstar));
    const uint16_t cand[4] = {plain, ds, half_next(ds, false), half_next(ds, true)};
    uint16_t best = plain;
    float best_e = 0.f;
    bool have = false;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if ((cand[c] & 0x7C00u) == 0x7C00u) continue;  // inf or nan
      const float d = __half2float(__ushort_as_half(cand[c]));
      const float inv = (d != 0.0f) ? __frcp_rn(d) : 0.0f;
      float e = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float r = __fmaf_rn(-d, static_cast<float>(q4_code(v[j], inv) - 8), v[j]);
        e = __fmaf_rn(__fmul_rn(om[j], r), r, e);
      }
      e = sum8(e);
      if (!have || e < best_e) {
        best = cand[c];
        best_e = e;
        have = true;
      }
    }
    const float dsel = __half2float(__ushort_as_half(best));
    store_block(v, dsel != 0.0f ? __frcp_rn(dsel) : 0.0f, best, t, ok, n, b, K, codes, scales, sums, expanded);
  }
}

// One thread per 18-byte block: fp16 scale then 16 code bytes, copied bit for
// bit, and the block's code sum sum_j (q_j - 8).
__global__ void __launch_bounds__(256) import_q4_0_kernel(const uint8_t* __restrict__ blocks, int64_t nblk,
                                                           uint8_t* __restrict__ codes,
                                                           uint16_t* __restrict__ scales,
                                                           int16_t* __restrict__ sums,
                                                           uint8_t* __restrict__ expanded) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= nblk) return;
  const uint16_t* src = reinterpret_cast<const uint16_t*>(blocks + i * 18);  // 2-byte aligned
  scales[i] = src[0];
  uint32_t q[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) q[j] = static_cast<uint32_t>(src[1 + 2 * j]) | (static_cast<uint32_t>(src[2 + 2 * j]) << 16);
  reinterpret_cast<uint4*>(codes)[i] = make_uint4(q[0], q[1], q[2], q[3]);
  int total = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t nib = (q[j] & 0x0F0F0F0Fu) + ((q[j] >> 4) & 0x0F0F0F0Fu);  // per byte <= 30
    total += static_cast<int>((nib & 0xFF) + ((nib >> 8) & 0xFF) + ((nib >> 16) & 0xFF) + (nib >> 24));
  }
  sums[i] = static_cast<int16_t>(total - 256);
  if (expanded) {  // blocks are row-major, so block i's 32 operand bytes sit at 32 i
    uint32_t e[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {  // word j: elements 4j..4j+3 (low nibbles), 16+4j.. (high)
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int byte = static_cast<int>((q[j] >> (8 * k)) & 0xFFu);
        lo |= e4m3_of_code(byte & 15) << (8 * k);
        hi |= e4m3_of_code(byte >> 4) << (8 * k);
      }
      e[j] = lo;
      e[4 + j] = hi;
    }
    uint4* dst = reinterpret_cast<uint4*>(expanded + i * 32);
    dst[0] = make_uint4(e[0], e[1], e[2], e[3]);
    dst[1] = make_uint4(e[4], e[5], e[6], e[7]);
  }
}

}  // namespace

// Rows rows .. round_up(rows, 8) - 1 of the expanded operand are zero (the GEMM
// loads 8-row groups).
cudaError_t zero_expanded_pad(uint8_t* expanded, int64_t rows, int64_t K, cudaStream_t stream) {
  if (!expanded) return cudaSuccess;
  const int64_t pad = ((rows + 7) / 8) * 8 - rows;
  if (pad == 0) return cudaSuccess;
  return cudaMemsetAsync(expanded + rows * K, 0, static_cast<size_t>(pad * K), stream);
}

cudaError_t launch_pack_q4_0(const void* w, int w_dtype, int64_t N, int64_t K, int64_t ldw, int rotate,
                             uint8_t* codes, uint16_t* scales, int16_t* sums, uint8_t* expanded,
                             cudaStream_t stream) {
  const int64_t ngroups = (N * (K / 32) + 3) / 4;
  int64_t ctas = (ngroups + 7) / 8;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  if (ctas > cap) ctas = cap;
  if (ctas < 1) ctas = 1;
  cudaError_t e = zero_expanded_pad(expanded, N, K, stream);
  if (e != cudaSuccess) return e;
  pack_q4_0_kernel<<<static_cast<unsigned>(ctas), 256, 0, stream>>>(w, w_dtype, N, K, ldw, rotate, codes, scales,
                                                                     sums, expanded);
  return cudaGetLastError();
}

cudaError_t launch_pack_q4_0_weighted(const void* w, int w_dtype, int64_t N, int64_t K, int64_t ldw, int rotate,
                                      const float* imp, uint8_t* codes, uint16_t* scales, int16_t* sums,
                                      uint8_t* expanded, cudaStream_t stream) {
  const int64_t ngroups = (N * (K / 32) + 3) / 4;
  int64_t ctas = (ngroups + 7) / 8;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 16;
  if (ctas > cap) ctas = cap;
  if (ctas < 1) ctas = 1;
  cudaError_t e = zero_expanded_pad(expanded, N, K, stream);
  if (e != cudaSuccess) return e;
  pack_q4_0_weighted_kernel<<<static_cast<unsigned>(ctas), 256, 0, stream>>>(w, w_dtype, N, K, ldw, rotate, imp, codes,
                                                                              scales, sums, expanded);
  return cudaGetLastError();
}

cudaError_t launch_import_q4_0(const void* blocks, int64_t N, int64_t K, uint8_t* codes, uint16_t* scales,
                               int16_t* sums, uint8_t* expanded, cudaStream_t stream) {
  const int64_t nblk = N * (K / 32);
  const int64_t ctas = (nblk + 255) / 256;
  cudaError_t e = zero_expanded_pad(expanded, N, K, stream);
  if (e != cudaSuccess) return e;
  import_q4_0_kernel<<<static_cast<unsigned>(ctas), 256, 0, stream>>>(static_cast<const uint8_t*>(blocks), nblk,
                                                                       codes, scales, sums, expanded);
  return cudaGetLastError();
}

}  // namespace w4a4
