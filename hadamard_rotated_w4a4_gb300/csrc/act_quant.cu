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
#include <cuda_bf16.h>

#include "w4a4_kernels.cuh"

namespace w4a4 {

namespace {

constexpr int kWarps = 8;
constexpr int kRow = 36;  // floats per padded block row in shared memory

// Stage h = 1 pairs the two halves of each register pair (scalar adds); stages
// h >= 2 pair whole register pairs, so each runs as paired fp32 adds -- the same
// IEEE additions in the same order, half the instructions.
__device__ __forceinline__ void fwht32(float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const float a = v[i], b = v[i + 1];
    v[i] = __fadd_rn(a, b);
    v[i + 1] = __fsub_rn(a, b);
  }
  float2 (&w)[16] = *reinterpret_cast<float2 (*)[16]>(&v);
#pragma unroll
  for (int h2 = 1; h2 < 16; h2 <<= 1) {  // h = 2 h2
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if ((j & h2) == 0) {
        const float2 a = w[j], b = w[j + h2];
        w[j] = __fadd2_rn(a, b);
        w[j + h2] = __fadd2_rn(a, make_float2(-b.x, -b.y));  // a - b, exactly
      }
    }
  }
}

// an already scaled value y * (1 / d): round half away from zero, clamp, and the
// 4-bit two's complement nibble
__device__ __forceinline__ uint32_t nib_scaled(float v) {
  float r = round_half_away(v);
  r = fminf(fmaxf(r, -8.0f), 7.0f);
  return static_cast<uint32_t>(static_cast<int>(r)) & 0xFu;
}

// One 32-element block held by this lane: rotate (optional), then
//   BITS = 4: d_a = amax / 7, int4 codes (round half away, clamp -8..7), 16
//             bytes in the Q4_0 nibble order; with `expanded`, also the 32
//             offset codes a + 8 as bytes in element order (the e4m3 operand
//             bytes of the dense GEMM);
//   BITS = 8: d_a = amax / 127, int8 codes (round half away, clamp -127..127),
//             32 bytes in element order (the exact path's activations);
//   BITS = 16: no quantisation (the rotate-only route): the 32 rotated values
//             as bf16, round to nearest even, 64 bytes in element order, no
//             scale;
// stored at block index i if ok.
__device__ __forceinline__ void rotate_block(float (&y)[32]) {
  fwht32(y);
  const float2 cst = make_float2(c_h32(), c_h32());
  float2 (&w)[16] = *reinterpret_cast<float2 (*)[16]>(&y);
#pragma unroll
  for (int k = 0; k < 16; ++k) w[k] = __fmul2_rn(w[k], cst);
}

// The int4 codes of an already scaled block, 3 or 4 instructions per value instead
// of the general rounding: when the maximum a is finite and nonzero and the
// reciprocal scale is finite, every |y| is at most 7 times (1 + a few ulp), so
// y + 1.5 * 2^23 lands in [2^23, 2^24), where the spacing is 1: the sum is
// 1.5 * 2^23 plus y rounded to the nearest integer (ties to even), and its low 4
// bits are that integer's two's complement nibble.  The result equals
// round-half-away-from-zero and the clamp to -8..7 unless some value sits exactly
// halfway between two integers (|y - nearest| = 0.5), or is NaN: then this returns
// false and the caller takes the general path.  Packs byte t = element t | element
// t + 16 << 4 into w.
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ bool pack_nibbles_fast(const float (&y)[32], float a, float inv, uint32_t (&w)[4]) {
  if (!(a > 0.0f && a <= 3.402823466e38f && inv <= 3.402823466e38f)) return false;
  constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
  const float2 (&yw)[16] = *reinterpret_cast<const float2 (*)[16]>(&y);
  uint32_t tb[32];
  float m = 0.0f;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const float2 t = __fadd2_rn(yw[k], make_float2(kMagic, kMagic));
    const float2 r = __fadd2_rn(t, make_float2(-kMagic, -kMagic));      // the nearest integer, exactly
    const float2 dd = __fadd2_rn(yw[k], make_float2(-r.x, -r.y));      // y - nearest, exactly
    m = max_nan(m, max_nan(fabsf(dd.x), fabsf(dd.y)));
    tb[2 * k] = __float_as_uint(t.x);
    tb[2 * k + 1] = __float_as_uint(t.y);
  }
  if (!(m < 0.5f)) return false;  // a tie (or a NaN): the general path decides
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint32_t lo = prmt(prmt(tb[4 * t], tb[4 * t + 1], 0x0040u), prmt(tb[4 * t + 2], tb[4 * t + 3], 0x0040u), 0x5410u);
    const uint32_t hi =
        prmt(prmt(tb[16 + 4 * t], tb[17 + 4 * t], 0x0040u), prmt(tb[18 + 4 * t], tb[19 + 4 * t], 0x0040u), 0x5410u);
    w[t] = (lo & 0x0F0F0F0Fu) | ((hi << 4) & 0xF0F0F0F0u);
  }
  return true;
}

template <int BITS>
__device__ __forceinline__ void quantize_block(float (&y)[32], int rotate, bool ok, uint8_t* __restrict__ codes,
                                               float* __restrict__ scales, uint8_t* __restrict__ expanded,
                                               int64_t i) {
  if (rotate) rotate_block(y);
  if constexpr (BITS == 16) {
    uint32_t w[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(y[2 * t], y[2 * t + 1]);  // .x = element 2t
      memcpy(&w[t], &h, 4);
    }
    if (ok) {
      uint4* dst = reinterpret_cast<uint4*>(codes) + 4 * i;
#pragma unroll
      for (int q = 0; q < 4; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    }
    return;
  }
  float a = 0.f;
#pragma unroll
  for (int k = 0; k < 32; ++k) a = fmaxf(a, fabsf(y[k]));
  if constexpr (BITS == 8) {
    const float d = __fdiv_rn(a, 127.0f);
    const float inv = (d != 0.0f) ? __frcp_rn(d) : 0.0f;
    uint32_t w[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      uint32_t word = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float r = round_half_away(__fmul_rn(y[4 * t + k], inv));
        r = fminf(fmaxf(r, -127.0f), 127.0f);
        word |= (static_cast<uint32_t>(static_cast<int>(r)) & 0xFFu) << (8 * k);
      }
      w[t] = word;
    }
    if (ok) {
      uint4* dst = reinterpret_cast<uint4*>(codes) + 2 * i;
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      scales[i] = d;
    }
    return;
  }
  const float d = __fdiv_rn(a, 7.0f);
  const float inv = (d != 0.0f) ? __frcp_rn(d) : 0.0f;
  {  // y * inv, paired (the same products)
    float2 (&yw)[16] = *reinterpret_cast<float2 (*)[16]>(&y);
    const float2 inv2 = make_float2(inv, inv);
#pragma unroll
    for (int k = 0; k < 16; ++k) yw[k] = __fmul2_rn(yw[k], inv2);
  }
  // byte t of the 16 = element t (low nibble) | element t + 16 (high nibble)
  uint32_t w[4];
  if (!pack_nibbles_fast(y, a, inv, w)) {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      uint32_t word = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t lo = nib_scaled(y[4 * t + k]);
        const uint32_t hi = nib_scaled(y[16 + 4 * t + k]);
        word |= (lo | (hi << 4)) << (8 * k);
      }
      w[t] = word;
    }
  }
  if (ok) {
    reinterpret_cast<uint4*>(codes)[i] = make_uint4(w[0], w[1], w[2], w[3]);
    scales[i] = d;
    if (expanded) {
      // a + 8 = nibble ^ 8; low nibbles are elements 0..15, high nibbles 16..31
      uint32_t u[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) u[t] = w[t] ^ 0x88888888u;
      uint4* dst = reinterpret_cast<uint4*>(expanded) + 2 * i;
      dst[0] = make_uint4(u[0] & 0x0F0F0F0Fu, u[1] & 0x0F0F0F0Fu, u[2] & 0x0F0F0F0Fu, u[3] & 0x0F0F0F0Fu);
      dst[1] = make_uint4((u[0] >> 4) & 0x0F0F0F0Fu, (u[1] >> 4) & 0x0F0F0F0Fu, (u[2] >> 4) & 0x0F0F0F0Fu,
                          (u[3] >> 4) & 0x0F0F0F0Fu);
    }
  }
}

template <int BITS>
__global__ void __launch_bounds__(32 * kWarps) act_rotate_quantize_kernel(const float* __restrict__ x, int64_t M,
                                                                          int64_t K, int64_t ldx, int rotate,
                                                                          uint8_t* __restrict__ codes,
                                                                          float* __restrict__ scales,
                                                                          uint8_t* __restrict__ expanded) {
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
    quantize_block<BITS>(y, rotate, ok, codes, scales, expanded, i);
  }
}

// ---------------------------------------------------------------------------
// Contiguous rows (ldx == K): the input is one array of M * B blocks of 128
// bytes.  Each warp streams its chunks of 32 blocks (4 KB) through a 3-deep
// ring of TMA loads (2D map [M*B][32 floats], 128-byte swizzle), the next
// chunk's load issued before the current one is computed, so every SM keeps
// up to 2 x 8 x 3 x 4 KB of reads in flight.  The swizzle puts 16-byte piece j
// of block row r at piece j ^ (r % 8): lane r reads its own block with eight
// conflict-free 16-byte loads, no transposition pass.
constexpr int kTmaWarps = 8;
#ifndef W4A4_ACT_STAGES
#define W4A4_ACT_STAGES 3
#endif
#ifndef W4A4_ACT_CTAS_PER_SM
#define W4A4_ACT_CTAS_PER_SM 2
#endif
constexpr int kTmaStages = W4A4_ACT_STAGES;
constexpr uint32_t kChunkBytes = 32 * 32 * sizeof(float);
constexpr uint64_t kActTimeoutNs = 1000000000ull;  // 1 s

struct __align__(1024) ActSmem {
  float buf[kTmaWarps][kTmaStages][32 * 32];
  uint64_t full[kTmaWarps][kTmaStages];
};

__device__ __forceinline__ uint32_t su32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t gtime() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false after 1 s (the caller records the error and winds down).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* b, uint32_t parity) {
  if (mbar_try(b, parity)) return true;
  const uint64_t t0 = gtime();
  while (!mbar_try(b, parity)) {
    if (gtime() - t0 > kActTimeoutNs) return false;
  }
  return true;
}
__device__ __forceinline__ void tma_load_chunk(float* dst, const CUtensorMap* map, int32_t row, uint64_t* bar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(bar)), "r"(kChunkBytes)
               : "memory");
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(su32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row), "r"(su32(bar))
      : "memory");
}

template <int BITS>
__global__ void __launch_bounds__(32 * kTmaWarps, W4A4_ACT_CTAS_PER_SM) act_rotate_quantize_tma_kernel(
    const __grid_constant__ CUtensorMap xmap, int64_t nblk, int rotate, uint8_t* __restrict__ codes,
    float* __restrict__ scales, uint8_t* __restrict__ expanded, int* err) {
  extern __shared__ __align__(1024) uint8_t act_smem[];
  ActSmem& S = *reinterpret_cast<ActSmem*>(act_smem);
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  if ((su32(act_smem) & 1023u) != 0) {  // the swizzle pattern assumes 1024-byte aligned stages; never expected
    if (threadIdx.x == 0 && err) atomicOr(err, 16);
    return;
  }
  // a GEMM launched after this kernel may start its set-up and weight loads now
  // (it waits for this grid to finish before it reads the activations)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t nchunks = (nblk + 31) / 32;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kTmaWarps + wib;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * kTmaWarps;
  const int64_t n_my = gw < nchunks ? (nchunks - gw + nw - 1) / nw : 0;
  if (lane == 0) {
    for (int st = 0; st < kTmaStages; ++st)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&S.full[wib][st])));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&xmap)) : "memory");
  }
  __syncwarp();
  int64_t issued = 0;  // meaningful in lane 0
  if (lane == 0) {
    for (; issued < n_my && issued < kTmaStages; ++issued)
      tma_load_chunk(S.buf[wib][issued], &xmap, static_cast<int32_t>((gw + issued * nw) * 32),
                     &S.full[wib][issued]);
  }
  bool failed = false;
  for (int64_t it = 0; it < n_my; ++it) {
    const int st = static_cast<int>(it % kTmaStages);
    if (!mbar_wait_bounded(&S.full[wib][st], static_cast<uint32_t>((it / kTmaStages) & 1))) {
      failed = true;
      break;
    }
    const float* row = S.buf[wib][st] + lane * 32;
    float y[32];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 v = *reinterpret_cast<const float4*>(row + 4 * (j ^ (lane & 7)));
      y[4 * j + 0] = v.x;
      y[4 * j + 1] = v.y;
      y[4 * j + 2] = v.z;
      y[4 * j + 3] = v.w;
    }
    // Before the stage is refilled by the TMA (the async proxy), every lane's
    // reads of it (the generic proxy) must have completed: the rotation consumes
    // all 32 values first, and the proxy fence orders the reads before the copy
    // lane 0 issues after the warp barrier.
    if (rotate) rotate_block(y);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0 && issued < n_my) {
      tma_load_chunk(S.buf[wib][st], &xmap, static_cast<int32_t>((gw + issued * nw) * 32), &S.full[wib][st]);
      ++issued;
    }
    const int64_t i = (gw + it * nw) * 32 + lane;
    quantize_block<BITS>(y, 0, i < nblk, codes, scales, expanded, i);
  }
  if (__any_sync(0xFFFFFFFFu, failed)) {
    // a load never completed: record it and wait (bounded) for the copies still
    // in flight, so that none lands after the block has exited
    if (lane == 0) {
      if (err) atomicOr(err, 8);
      for (int64_t it = issued > kTmaStages ? issued - kTmaStages : 0; it < issued; ++it)
        mbar_wait_bounded(&S.full[wib][it % kTmaStages], static_cast<uint32_t>((it / kTmaStages) & 1));
    }
    __syncwarp();
  }
}

}  // namespace

namespace {
template <int BITS>
cudaError_t launch_act(const float* x, int64_t M, int64_t K, int64_t ldx, int rotate, uint8_t* codes, float* scales,
                       uint8_t* expanded, cudaStream_t stream) {
  const int64_t nblk = M * (K / 32);
  const int64_t nchunks = (nblk + 31) / 32;
  if (ldx == K && nblk < (int64_t(1) << 31) - 64) {
    CUtensorMap xmap;
    cudaError_t e = encode_2d_map(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, x, 32, static_cast<uint64_t>(nblk),
                                  32 * sizeof(float), 32, 32, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e == cudaSuccess) {
      static bool configured[64] = {};
      int dev = 0;
      cudaGetDevice(&dev);
      if (dev >= 0 && dev < 64 && !configured[dev]) {
        e = cudaFuncSetAttribute(act_rotate_quantize_tma_kernel<BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(sizeof(ActSmem)));
        if (e != cudaSuccess) return e;
        configured[dev] = true;
      }
      int64_t ctas = (nchunks + kTmaWarps - 1) / kTmaWarps;
      const int64_t cap = static_cast<int64_t>(num_sms()) * W4A4_ACT_CTAS_PER_SM;
      if (ctas > cap) ctas = cap;
      if (ctas < 1) ctas = 1;
      act_rotate_quantize_tma_kernel<BITS><<<static_cast<unsigned>(ctas), 32 * kTmaWarps, sizeof(ActSmem), stream>>>(
          xmap, nblk, rotate, codes, scales, expanded, device_error_word());
      return cudaGetLastError();
    }
  }
  int64_t ctas = (nchunks + kWarps - 1) / kWarps;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 4;  // 4 x 256 threads per SM
  if (ctas > cap) ctas = cap;
  if (ctas < 1) ctas = 1;
  act_rotate_quantize_kernel<BITS><<<static_cast<unsigned>(ctas), 32 * kWarps, 0, stream>>>(x, M, K, ldx, rotate, codes,
                                                                                       scales, expanded);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_act_rotate_quantize(const float* x, int64_t M, int64_t K, int64_t ldx, int rotate,
                                       uint8_t* codes, float* scales, uint8_t* expanded, cudaStream_t stream) {
  return launch_act<4>(x, M, K, ldx, rotate, codes, scales, expanded, stream);
}

cudaError_t launch_act_rotate_quantize8(const float* x, int64_t M, int64_t K, int64_t ldx, int rotate,
                                        int8_t* codes, float* scales, cudaStream_t stream) {
  return launch_act<8>(x, M, K, ldx, rotate, reinterpret_cast<uint8_t*>(codes), scales, nullptr, stream);
}

cudaError_t launch_act_rotate_bf16(const float* x, int64_t M, int64_t K, int64_t ldx, int rotate, uint16_t* out,
                                   cudaStream_t stream) {
  return launch_act<16>(x, M, K, ldx, rotate, reinterpret_cast<uint8_t*>(out), nullptr, nullptr, stream);
}

}  // namespace w4a4
