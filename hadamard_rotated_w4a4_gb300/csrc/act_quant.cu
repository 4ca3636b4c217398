// Activation rotate + int4 quantise (engine docs "The lean option: ROCmFP4,
// ROCmI4 and Hadamard Q4_0", section "Hadamard-rotated Q4_0: W4A4 prompt
// processing": the activations get the weights' per-32-block rotation and are
// rounded to 4 bits per block).
//
// HBM-bound streaming kernel, written to stay under the instruction budget of
// the memory system (about 20 warp instructions per 128-byte block at full HBM
// rate): one lane owns one 32-element block, so the butterfly, the block
// maximum and the scale are computed once per block, in registers, with no
// shuffles.  A warp takes 32 consecutive blocks (flat index over rows x blocks);
// it reads them with 16-byte loads that are coalesced across the warp (each
// instruction covers 512 contiguous bytes of 4 blocks), transposes through a
// padded shared-memory tile (144-byte rows: the 16-byte accesses of 8 lanes hit
// distinct banks) and writes back 16 code bytes and one scale per lane, again
// contiguous across the warp.
//
// Butterfly order: stages h = 1, 2, 4, 8, 16, pairs (i, i + h) -> (a + b, a - b),
// then one multiply by fl32(1/sqrt 32) -- the fp32 evaluation order the
// quantiser's decisions are defined on.
#include "w4a4_kernels.cuh"

namespace w4a4 {

namespace {

constexpr int kWarps = 8;
constexpr int kRow = 36;  // floats per padded block row in shared memory

__device__ __forceinline__ void fwht32(float (&v)[32]) {
#pragma unroll
  for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = __fadd_rn(a, b);
        v[i + h] = __fsub_rn(a, b);
      }
    }
  }
}

// round half away from zero, then to a 4-bit two's complement nibble
__device__ __forceinline__ uint32_t nib(float y, float inv) {
  float r = round_half_away(__fmul_rn(y, inv));
  r = fminf(fmaxf(r, -8.0f), 7.0f);
  return static_cast<uint32_t>(static_cast<int>(r)) & 0xFu;
}

__global__ void __launch_bounds__(32 * kWarps) act_rotate_quantize_kernel(const float* __restrict__ x, int64_t M,
                                                                          int64_t K, int64_t ldx, int rotate,
                                                                          uint8_t* __restrict__ codes,
                                                                          float* __restrict__ scales) {
  __shared__ __align__(16) float tile[kWarps][32 * kRow];
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  float* T = tile[wib];
  const int64_t B = K / 32;
  const int64_t nblk = M * B;
  const int64_t nchunks = (nblk + 31) / 32;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarps + wib;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * kWarps;

  for (int64_t c = gw; c < nchunks; c += nw) {
    // this lane's block and the address of its 32 floats
    const int64_t i = c * 32 + lane;
    const bool ok = i < nblk;
    const int64_t m = ok ? i / B : 0;
    const int64_t b = ok ? i - m * B : 0;
    const float* src = x + m * ldx + b * 32;
    // cooperative, coalesced load: instruction j brings float4 (lane & 7) of block 4j + lane / 8
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int blk = 4 * j + (lane >> 3);
      const unsigned long long sa =
          __shfl_sync(0xFFFFFFFFu, reinterpret_cast<unsigned long long>(src), blk);
      const bool bok = c * 32 + blk < nblk;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (bok) v = __ldcs(reinterpret_cast<const float4*>(sa) + (lane & 7));
      *reinterpret_cast<float4*>(T + blk * kRow + 4 * (lane & 7)) = v;
    }
    __syncwarp();
    float y[32];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float4 v = *reinterpret_cast<const float4*>(T + lane * kRow + 4 * k);
      y[4 * k + 0] = v.x;
      y[4 * k + 1] = v.y;
      y[4 * k + 2] = v.z;
      y[4 * k + 3] = v.w;
    }
    __syncwarp();
    if (rotate) {
      fwht32(y);
      const float cst = c_h32();
#pragma unroll
      for (int k = 0; k < 32; ++k) y[k] = __fmul_rn(y[k], cst);
    }
    float a = 0.f;
#pragma unroll
    for (int k = 0; k < 32; ++k) a = fmaxf(a, fabsf(y[k]));
    const float d = __fdiv_rn(a, 7.0f);
    const float inv = (d != 0.0f) ? __frcp_rn(d) : 0.0f;
    // byte t of the 16 = element t (low nibble) | element t + 16 (high nibble)
    uint32_t w[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      uint32_t word = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t lo = nib(y[4 * t + k], inv);
        const uint32_t hi = nib(y[16 + 4 * t + k], inv);
        word |= (lo | (hi << 4)) << (8 * k);
      }
      w[t] = word;
    }
    if (ok) {
      reinterpret_cast<uint4*>(codes)[i] = make_uint4(w[0], w[1], w[2], w[3]);
      scales[i] = d;
    }
  }
}

}  // namespace

cudaError_t launch_act_rotate_quantize(const float* x, int64_t M, int64_t K, int64_t ldx, int rotate,
                                       uint8_t* codes, float* scales, cudaStream_t stream) {
  const int64_t nchunks = (M * (K / 32) + 31) / 32;
  int64_t ctas = (nchunks + kWarps - 1) / kWarps;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 4;  // 4 x 256 threads per SM
  if (ctas > cap) ctas = cap;
  if (ctas < 1) ctas = 1;
  act_rotate_quantize_kernel<<<static_cast<unsigned>(ctas), 32 * kWarps, 0, stream>>>(x, M, K, ldx, rotate, codes,
                                                                                       scales);
  return cudaGetLastError();
}

}  // namespace w4a4
