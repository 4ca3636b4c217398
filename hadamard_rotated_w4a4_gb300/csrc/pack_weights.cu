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

__global__ void __launch_bounds__(256) pack_q4_0_kernel(const void* __restrict__ w, int w_dtype, int64_t N,
                                                         int64_t K, int64_t ldw, int rotate,
                                                         uint8_t* __restrict__ codes,
                                                         uint16_t* __restrict__ scales,
                                                         int16_t* __restrict__ sums) {
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
    float v[4] = {0.f, 0.f, 0.f, 0.f};
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
    // signed value of largest magnitude, lowest index on ties
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
    const float d = __fdiv_rn(mval, -8.0f);
    const float inv = (d != 0.0f) ? __frcp_rn(d) : 0.0f;
    uint32_t lo = 0;
    int qsum = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float r = round_half_away(__fmul_rn(v[j], inv));
      r = fminf(fmaxf(__fadd_rn(r, 8.0f), 0.0f), 15.0f);
      const int q = static_cast<int>(r);
      lo |= static_cast<uint32_t>(q) << (8 * j);
      qsum += q - 8;
    }
    qsum += __shfl_xor_sync(0xFFFFFFFFu, qsum, 1);
    qsum += __shfl_xor_sync(0xFFFFFFFFu, qsum, 2);
    qsum += __shfl_xor_sync(0xFFFFFFFFu, qsum, 4);
    const uint32_t hi = __shfl_down_sync(0xFFFFFFFFu, lo << 4, 4);
    if (ok) {
      if (t < 4) reinterpret_cast<uint32_t*>(codes + n * (K / 2) + b * 16)[t] = lo | hi;
      if (t == 0) {
        scales[n * B + b] = __half_as_ushort(__float2half_rn(d));
        sums[n * B + b] = static_cast<int16_t>(qsum);
      }
    }
  }
}

// One thread per 18-byte block: fp16 scale then 16 code bytes, copied bit for
// bit, and the block's code sum sum_j (q_j - 8).
__global__ void __launch_bounds__(256) import_q4_0_kernel(const uint8_t* __restrict__ blocks, int64_t nblk,
                                                           uint8_t* __restrict__ codes,
                                                           uint16_t* __restrict__ scales,
                                                           int16_t* __restrict__ sums) {
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
}

}  // namespace

cudaError_t launch_pack_q4_0(const void* w, int w_dtype, int64_t N, int64_t K, int64_t ldw, int rotate,
                             uint8_t* codes, uint16_t* scales, int16_t* sums, cudaStream_t stream) {
  const int64_t ngroups = (N * (K / 32) + 3) / 4;
  int64_t ctas = (ngroups + 7) / 8;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  if (ctas > cap) ctas = cap;
  if (ctas < 1) ctas = 1;
  pack_q4_0_kernel<<<static_cast<unsigned>(ctas), 256, 0, stream>>>(w, w_dtype, N, K, ldw, rotate, codes, scales,
                                                                     sums);
  return cudaGetLastError();
}

cudaError_t launch_import_q4_0(const void* blocks, int64_t N, int64_t K, uint8_t* codes, uint16_t* scales,
                               int16_t* sums, cudaStream_t stream) {
  const int64_t nblk = N * (K / 32);
  const int64_t ctas = (nblk + 255) / 256;
  import_q4_0_kernel<<<static_cast<unsigned>(ctas), 256, 0, stream>>>(static_cast<const uint8_t*>(blocks), nblk,
                                                                       codes, scales, sums);
  return cudaGetLastError();
}

}  // namespace w4a4
