// Activation rotate + int4 quantise (engine docs "The lean option: ROCmFP4,
// ROCmI4 and Hadamard Q4_0", section "Hadamard-rotated Q4_0: W4A4 prompt
// processing": the activations get the weights' per-32-block rotation and are
// rounded to 4 bits per block).
//
// HBM-bound streaming kernel.  Eight lanes own one 32-element block (a 16-byte
// fp32 vector each), so a warp reads 4 blocks = 512 contiguous bytes per load.
// The 32-point butterfly runs its first two stages (h = 1, 2) inside each
// lane's four values and the last three (h = 4, 8, 16) across lanes with
// shuffles, in that order, matching the fp32 evaluation order the quantiser's
// decisions are defined on.  Each warp keeps two groups of 4 blocks in flight.
#include "w4a4_kernels.cuh"

namespace w4a4 {

namespace {

struct Blk {
  float4 v;
  int64_t m, b;
  bool ok;
};

__device__ __forceinline__ void butterfly_in_lane(float4& v) {
  // h = 1: (0,1), (2,3)
  float a0 = __fadd_rn(v.x, v.y), a1 = __fsub_rn(v.x, v.y);
  float a2 = __fadd_rn(v.z, v.w), a3 = __fsub_rn(v.z, v.w);
  // h = 2: (0,2), (1,3)
  v.x = __fadd_rn(a0, a2);
  v.z = __fsub_rn(a0, a2);
  v.y = __fadd_rn(a1, a3);
  v.w = __fsub_rn(a1, a3);
}

__device__ __forceinline__ float bfly_xlane(float v, int lane_bit, bool upper) {
  const float o = __shfl_xor_sync(0xFFFFFFFFu, v, lane_bit);
  // lower lane keeps a + b, upper lane keeps a - b (a = lower's value)
  return upper ? __fsub_rn(o, v) : __fadd_rn(v, o);
}

__device__ __forceinline__ void butterfly_across_lanes(float4& v, int t) {
#pragma unroll
  for (int s = 0; s < 3; ++s) {  // h = 4, 8, 16  <->  lane bit 1, 2, 4 within the 8-lane group
    const int bit = 1 << s;
    const bool up = (t & bit) != 0;
    v.x = bfly_xlane(v.x, bit, up);
    v.y = bfly_xlane(v.y, bit, up);
    v.z = bfly_xlane(v.z, bit, up);
    v.w = bfly_xlane(v.w, bit, up);
  }
}

__device__ __forceinline__ uint32_t q_nib(float y, float inv) {
  float r = round_half_away(__fmul_rn(y, inv));
  r = fminf(fmaxf(r, -8.0f), 7.0f);
  return static_cast<uint32_t>(static_cast<int>(r)) & 0xFu;
}

__device__ __forceinline__ void quantize_store(const Blk& k, int t, bool rotate, int64_t K, uint8_t* codes,
                                               float* scales) {
  float4 y = k.v;
  if (rotate) {
    butterfly_in_lane(y);
    butterfly_across_lanes(y, t);
    const float c = c_h32();
    y.x = __fmul_rn(y.x, c);
    y.y = __fmul_rn(y.y, c);
    y.z = __fmul_rn(y.z, c);
    y.w = __fmul_rn(y.w, c);
  }
  float a = fmaxf(fmaxf(fabsf(y.x), fabsf(y.y)), fmaxf(fabsf(y.z), fabsf(y.w)));
  a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
  a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
  a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 4));
  const float d = __fdiv_rn(a, 7.0f);
  const float inv = (d != 0.0f) ? __frcp_rn(d) : 0.0f;
  const uint32_t n0 = q_nib(y.x, inv), n1 = q_nib(y.y, inv), n2 = q_nib(y.z, inv), n3 = q_nib(y.w, inv);
  // Byte i of the block = element i (low nibble) | element i + 16 (high nibble).
  // Lane t < 4 holds elements 4t..4t+3 (low halves of bytes 4t..4t+3); lane t + 4
  // holds elements 16 + 4t.. (their high halves).
  const uint32_t lo = n0 | (n1 << 8) | (n2 << 16) | (n3 << 24);
  const uint32_t hi = __shfl_down_sync(0xFFFFFFFFu, lo << 4, 4);
  if (k.ok) {
    if (t < 4) {
      uint32_t* dst = reinterpret_cast<uint32_t*>(codes + k.m * (K / 2) + k.b * 16) + t;
      *dst = lo | hi;
    }
    if (t == 0) scales[k.m * (K / 32) + k.b] = d;
  }
}

__device__ __forceinline__ Blk load_blk(const float* __restrict__ x, int64_t g, int sub, int t, int64_t nblk,
                                        int64_t B, int64_t ldx) {
  Blk k;
  const int64_t idx = g * 4 + sub;
  k.ok = idx < nblk;
  k.m = k.ok ? idx / B : 0;
  k.b = k.ok ? idx - k.m * B : 0;
  if (k.ok) {
    const float4* p = reinterpret_cast<const float4*>(x + k.m * ldx + k.b * 32) + t;
    k.v = __ldcs(p);  // streamed once: evict-first
  } else {
    k.v = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  return k;
}

__global__ void __launch_bounds__(256) act_rotate_quantize_kernel(const float* __restrict__ x, int64_t M,
                                                                   int64_t K, int64_t ldx, int rotate,
                                                                   uint8_t* __restrict__ codes,
                                                                   float* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int sub = lane >> 3;  // which of the warp's 4 blocks
  const int t = lane & 7;     // which 16-byte quarter of the block
  const int64_t B = K / 32;
  const int64_t nblk = M * B;
  const int64_t ngroups = (nblk + 3) / 4;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t g = warp; g < ngroups; g += 2 * nwarps) {
    const int64_t g2 = g + nwarps;
    Blk k0 = load_blk(x, g, sub, t, nblk, B, ldx);
    Blk k1 = load_blk(x, g2, sub, t, nblk, B, ldx);
    quantize_store(k0, t, rotate != 0, K, codes, scales);
    if (g2 < ngroups) quantize_store(k1, t, rotate != 0, K, codes, scales);  // warp-uniform
  }
}

}  // namespace

cudaError_t launch_act_rotate_quantize(const float* x, int64_t M, int64_t K, int64_t ldx, int rotate,
                                       uint8_t* codes, float* scales, cudaStream_t stream) {
  const int64_t nblk = M * (K / 32);
  const int64_t ngroups = (nblk + 3) / 4;
  const int threads = 256;
  const int64_t warps_needed = (ngroups + 1) / 2;
  int64_t ctas = (warps_needed + 7) / 8;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;  // 8 CTAs x 256 threads fill an SM
  if (ctas > cap) ctas = cap;
  if (ctas < 1) ctas = 1;
  act_rotate_quantize_kernel<<<static_cast<unsigned>(ctas), threads, 0, stream>>>(x, M, K, ldx, rotate, codes,
                                                                                   scales);
  return cudaGetLastError();
}

}  // namespace w4a4
