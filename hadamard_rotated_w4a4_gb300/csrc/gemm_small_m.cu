// Block-scaled W4A4 product for small token batches (M <= 8): verification
// batches of a drafter (engine docs "The lean option: ROCmFP4, ROCmI4 and
// Hadamard Q4_0", a row-tiled Q4_0 kernel for 8-column verification batches:
// each weight is unpacked once for all columns, and the output is bit for bit
// that of the general kernel).
//
// With M <= 8 the product is a weight stream, too narrow for the 5th-gen tensor
// core tile.  Here each block's integer dot products run on the warp-level f16
// tensor core: mma.sync m16n8k16, A = 16 weight rows, B = the 8 token columns.
// A code nibble n placed under the f16 exponent byte 0x64 (prmt) is the f16
// 1024 + n, and one exact f16x2 subtraction of 1032 leaves n - 8: q - 8 for a
// weight code q, and the signed a for an activation nibble flipped by ^ 8.
// Every product and partial sum is an integer below 2^12, so the two MMAs of a
// block (its two K halves) give D = P exactly in fp32.
//
// A CTA owns 16 weight rows; its 4 warps split K round robin in chunks of 8
// blocks (warp w takes chunks w, w + 4, ...).  Each warp streams its chunks'
// weight codes and scales and the token rows' codes and scales into its own
// three-stage shared-memory ring with cp.async, and computes each block's
// t = round(d_w P) for its 16 rows x 8 tokens ahead of time.  The fold
// acc = fma(t, d_a, acc) is the general kernel's chain in K order: the
// accumulators pass from the warp that folded chunk c to the warp of chunk
// c + 1 through shared memory and a named barrier (bar.arrive / bar.sync, two
// warps), so against the general kernel's whole-tile schedule the results agree
// bit for bit and no output depends on M or on the other tokens.
#include <cuda_fp16.h>

#include "w4a4_kernels.cuh"

namespace w4a4 {

namespace {

constexpr int kSmMaxM = 8;
constexpr int kSmWarps = 4;                 // the K split
constexpr int kSmRows = 16;                 // weight rows per CTA (the MMA's M)
constexpr int kSmChunk = 8;                 // blocks per chunk
constexpr int kSmStages = 3;                // per-warp ring: two chunks in flight
constexpr int kSmCtasPerSm = 3;             // 16-row tiles resident at once: 456 on 152 SMs
constexpr int kRowB = kSmChunk * 16 + 16;   // code bytes per row and stage (144: rows 4 banks apart)
constexpr int kWsRow = kSmChunk + 8;        // fp16 weight scales per row and stage (32 B: one 16-byte load)
constexpr int kAsRow = kSmChunk + 4;        // fp32 activation scales per token and stage (48 B)

struct WarpStage {
  uint8_t w[kSmRows][kRowB];     // weight codes, 16 rows x 8 blocks
  uint8_t a[kSmMaxM][kRowB];     // activation codes, 8 tokens x 8 blocks
  uint16_t ws[kSmRows][kWsRow];  // weight scales d_w (fp16 bits)
  float as[kSmMaxM][kAsRow];     // activation scales d_a
};
static_assert(sizeof(WarpStage) % 16 == 0, "stages stay 16-byte aligned");

struct SmallMSmem {
  WarpStage st[kSmWarps][kSmStages];
  float4 hand[32];  // the fold's accumulators, passed from warp to warp
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Named barriers 1..4 between two warps: the warp that folded chunk c arrives,
// the warp of chunk c + 1 waits.
__device__ __forceinline__ void bar_arrive(int id) { asm volatile("bar.arrive %0, 64;" ::"r"(id) : "memory"); }
__device__ __forceinline__ void bar_wait(int id) { asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory"); }

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
// f16x2 (n0 - 8, n1 - 8) of the nibbles in the two bytes `sel` picks from x
// (bytes holding one nibble each): the byte under the exponent byte 0x64 is
// 1024 + n, minus 1032 exactly.
__device__ __forceinline__ uint32_t nib_pair_f16(uint32_t x, uint32_t sel) {
  const uint32_t h = prmt(x, 0x64646464u, sel);
  __half2 a, b;
  const uint32_t c = 0x64086408u;
  memcpy(&a, &h, 4);
  memcpy(&b, &c, 4);
  const __half2 r = __hsub2(a, b);
  uint32_t out;
  memcpy(&out, &r, 4);
  return out;
}
// D += A B, m16n8k16, f16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// D = A B (no accumulator input).
__device__ __forceinline__ void mma_f16_first(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

struct SmallMArgs {
  const uint8_t* w_codes;
  const uint16_t* w_scales;
  const uint8_t* a_codes;
  const float* a_scales;
  int64_t N, K;
  int M;
  bool ws16;  // weight-scale rows copy in 16-byte pieces (B % 8 == 0, 16-byte base)
  bool as16;  // activation-scale rows copy in 16-byte pieces (B % 4 == 0, 16-byte base)
};

// Copy chunk [b0, b0 + nb) of the CTA's 16 weight rows and the M token rows
// into stage s (one warp).  Rows past N and tokens past M are not copied; the
// values computed from them are never stored.
__device__ __forceinline__ void load_stage(WarpStage& s, const SmallMArgs& p, int64_t n0, int64_t b0, int nb,
                                           int lane) {
  const int64_t B = p.K / 32, rowb = p.K / 2;
#pragma unroll
  for (int i = 0; i < kSmRows * kSmChunk / 32; ++i) {  // 4 pieces of 16 code bytes per lane
    const int pc = lane + 32 * i, r = pc / kSmChunk, bb = pc % kSmChunk;
    if (bb < nb && n0 + r < p.N) cp_async16(&s.w[r][bb * 16], p.w_codes + (n0 + r) * rowb + (b0 + bb) * 16);
  }
#pragma unroll
  for (int i = 0; i < kSmMaxM * kSmChunk / 32; ++i) {  // 2 per lane
    const int pc = lane + 32 * i, r = pc / kSmChunk, bb = pc % kSmChunk;
    if (bb < nb && r < p.M) cp_async16(&s.a[r][bb * 16], p.a_codes + r * rowb + (b0 + bb) * 16);
  }
  if (p.ws16) {  // 16 rows x 1 piece of 8 scales
    const int r = lane;
    if (r < kSmRows && n0 + r < p.N) cp_async16(&s.ws[r][0], p.w_scales + (n0 + r) * B + b0);
  } else if (lane < nb) {
#pragma unroll
    for (int r = 0; r < kSmRows; ++r)
      if (n0 + r < p.N) s.ws[r][lane] = p.w_scales[(n0 + r) * B + b0 + lane];
  }
  if (p.as16) {  // 8 tokens x 2 pieces of 4 scales
    const int r = lane >> 1, q = lane & 1;
    if (r < p.M && q * 4 < nb) cp_async16(&s.as[r][q * 4], p.a_scales + r * B + b0 + q * 4);
  } else if (lane < nb) {
#pragma unroll
    for (int r = 0; r < kSmMaxM; ++r)
      if (r < p.M) s.as[r][lane] = p.a_scales[r * B + b0 + lane];
  }
}

__global__ void __launch_bounds__(32 * kSmWarps, kSmCtasPerSm) w4a4_small_m_kernel(SmallMArgs p, float* __restrict__ y, int64_t ldy) {
  extern __shared__ __align__(16) uint8_t sm_raw[];
  SmallMSmem& S = *reinterpret_cast<SmallMSmem*>(sm_raw);
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  const int g = lane >> 2, tq = lane & 3;  // MMA fragment coordinates
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kSmRows;
  const int64_t B = p.K / 32;
  const int nchunks = static_cast<int>((B + kSmChunk - 1) / kSmChunk);
  const int mine = w < nchunks ? (nchunks - w + kSmWarps - 1) / kSmWarps : 0;  // chunks w, w + 4, ...
  auto chunk_len = [&](int c) {
    const int64_t left = B - static_cast<int64_t>(c) * kSmChunk;
    return static_cast<int>(left < kSmChunk ? left : kSmChunk);
  };
  WarpStage* ring = S.st[w];

  for (int i = 0; i < kSmStages - 1; ++i) {
    const int c = w + kSmWarps * i;
    if (i < mine) load_stage(ring[i], p, n0, static_cast<int64_t>(c) * kSmChunk, chunk_len(c), lane);
    cp_async_commit();
  }
  float2 acc01 = make_float2(0.f, 0.f), acc23 = make_float2(0.f, 0.f);  // rows g, g + 8 x tokens 2tq, 2tq + 1
  for (int i = 0; i < mine; ++i) {
    const int c = w + kSmWarps * i;
    {  // this warp's chunk two ahead streams into the stage chunk i - 1 used
      const int inext = i + kSmStages - 1;
      if (inext < mine) {
        const int cn = w + kSmWarps * inext;
        load_stage(ring[inext % kSmStages], p, n0, static_cast<int64_t>(cn) * kSmChunk, chunk_len(cn), lane);
      }
      cp_async_commit();
    }
    cp_async_wait<kSmStages - 1>();
    __syncwarp();
    const WarpStage& s = ring[i % kSmStages];
    const int nb = chunk_len(c);
    // t = round(d_w P) for every block of the chunk, before the fold's turn comes
    float2 t01[kSmChunk], t23[kSmChunk];  // rows g and g + 8, tokens (2tq, 2tq + 1)
    const uint32_t* w_lo = reinterpret_cast<const uint32_t*>(&s.w[g][0]) + tq;
    const uint32_t* w_hi = reinterpret_cast<const uint32_t*>(&s.w[g + 8][0]) + tq;
    const uint32_t* a_r = reinterpret_cast<const uint32_t*>(&s.a[g][0]) + tq;
    const uint4 dwv0 = *reinterpret_cast<const uint4*>(&s.ws[g][0]);      // 8 fp16 d_w of row g
    const uint4 dwv1 = *reinterpret_cast<const uint4*>(&s.ws[g + 8][0]);  // and of row g + 8
    const uint32_t dw0w[4] = {dwv0.x, dwv0.y, dwv0.z, dwv0.w}, dw1w[4] = {dwv1.x, dwv1.y, dwv1.z, dwv1.w};
    constexpr uint32_t kLow = 0x0F0F0F0Fu;
    auto block_t = [&](int bb) {
      const uint32_t x0 = w_lo[bb * 4], x1 = w_hi[bb * 4];
      const uint32_t xa = a_r[bb * 4] ^ 0x88888888u;  // a + 8 in every nibble
      const uint32_t l0 = x0 & kLow, h0 = (x0 >> 4) & kLow, l1 = x1 & kLow, h1 = (x1 >> 4) & kLow;
      const uint32_t la = xa & kLow, ha = (xa >> 4) & kLow;
      // k 4tq..4tq+3 (low nibbles) in the first K half, k 16+4tq.. (high) in the
      // second; in each, byte pair (0, 1) -> k slots 2tq, 2tq+1, (2, 3) -> 2tq+8, 2tq+9
      const uint32_t b1a = nib_pair_f16(la, 0x4140u), b1b = nib_pair_f16(la, 0x4342u);
      const uint32_t b2a = nib_pair_f16(ha, 0x4140u), b2b = nib_pair_f16(ha, 0x4342u);
      float d[4];
      mma_f16_first(d, nib_pair_f16(l0, 0x4140u), nib_pair_f16(l1, 0x4140u), nib_pair_f16(l0, 0x4342u),
                    nib_pair_f16(l1, 0x4342u), b1a, b1b);
      mma_f16(d, nib_pair_f16(h0, 0x4140u), nib_pair_f16(h1, 0x4140u), nib_pair_f16(h0, 0x4342u),
              nib_pair_f16(h1, 0x4342u), b2a, b2b);
      const float dw0 = __half2float(__ushort_as_half(static_cast<unsigned short>(dw0w[bb >> 1] >> (16 * (bb & 1)))));
      const float dw1 = __half2float(__ushort_as_half(static_cast<unsigned short>(dw1w[bb >> 1] >> (16 * (bb & 1)))));
      t01[bb] = __fmul2_rn(make_float2(d[0], d[1]), make_float2(dw0, dw0));
      t23[bb] = __fmul2_rn(make_float2(d[2], d[3]), make_float2(dw1, dw1));
    };
    const bool full = nb == kSmChunk;  // every chunk but a ragged last one: no per-block tests
    if (full) {
#pragma unroll
      for (int bb = 0; bb < kSmChunk; ++bb) block_t(bb);
    } else {
#pragma unroll
      for (int bb = 0; bb < kSmChunk; ++bb)
        if (bb < nb) block_t(bb);
    }
    float2 da[kSmChunk];  // d_a of tokens (2tq, 2tq + 1)
    {
      const float4 p0 = *reinterpret_cast<const float4*>(&s.as[2 * tq][0]);
      const float4 p1 = *reinterpret_cast<const float4*>(&s.as[2 * tq][4]);
      const float4 q0 = *reinterpret_cast<const float4*>(&s.as[2 * tq + 1][0]);
      const float4 q1 = *reinterpret_cast<const float4*>(&s.as[2 * tq + 1][4]);
      da[0] = make_float2(p0.x, q0.x); da[1] = make_float2(p0.y, q0.y);
      da[2] = make_float2(p0.z, q0.z); da[3] = make_float2(p0.w, q0.w);
      da[4] = make_float2(p1.x, q1.x); da[5] = make_float2(p1.y, q1.y);
      da[6] = make_float2(p1.z, q1.z); da[7] = make_float2(p1.w, q1.w);
    }
    __syncwarp();  // every lane is done with the stage before it is refilled
    // the fold, in K order: chunk c continues the accumulators of chunk c - 1
    if (c > 0) {
      bar_wait(1 + w);
      const float4 h = S.hand[lane];
      acc01 = make_float2(h.x, h.y);
      acc23 = make_float2(h.z, h.w);
    }
    // each lane of the f32x2 FMA rounds as fmaf
    if (full) {
#pragma unroll
      for (int bb = 0; bb < kSmChunk; ++bb) {
        acc01 = __ffma2_rn(t01[bb], da[bb], acc01);
        acc23 = __ffma2_rn(t23[bb], da[bb], acc23);
      }
    } else {
#pragma unroll
      for (int bb = 0; bb < kSmChunk; ++bb) {
        if (bb < nb) {
          acc01 = __ffma2_rn(t01[bb], da[bb], acc01);
          acc23 = __ffma2_rn(t23[bb], da[bb], acc23);
        }
      }
    }
    if (c + 1 < nchunks) {
      S.hand[lane] = make_float4(acc01.x, acc01.y, acc23.x, acc23.y);
      __threadfence_block();
      bar_arrive(1 + (w + 1) % kSmWarps);
    } else {  // the last chunk: this warp holds the finished sums
      const int m0 = 2 * tq;
      const int64_t r0 = n0 + g, r1 = n0 + g + 8;
      if (m0 < p.M) {
        if (r0 < p.N) y[static_cast<int64_t>(m0) * ldy + r0] = acc01.x;
        if (r1 < p.N) y[static_cast<int64_t>(m0) * ldy + r1] = acc23.x;
      }
      if (m0 + 1 < p.M) {
        if (r0 < p.N) y[static_cast<int64_t>(m0 + 1) * ldy + r0] = acc01.y;
        if (r1 < p.N) y[static_cast<int64_t>(m0 + 1) * ldy + r1] = acc23.y;
      }
    }
  }
  cp_async_wait<0>();
}

}  // namespace

cudaError_t launch_gemm_small_m(const uint8_t* w_codes, const uint16_t* w_scales, int64_t N, const uint8_t* a_codes,
                                const float* a_scales, int M, int64_t K, float* y, int64_t ldy, cudaStream_t stream) {
  if (M < 1 || M > kSmMaxM || K < 32) return cudaErrorInvalidValue;
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
  const int64_t B = K / 32;
  SmallMArgs p{w_codes, w_scales, a_codes, a_scales, N, K, M,
               B % 8 == 0 && reinterpret_cast<uintptr_t>(w_scales) % 16 == 0,
               B % 4 == 0 && reinterpret_cast<uintptr_t>(a_scales) % 16 == 0};
  w4a4_small_m_kernel<<<static_cast<unsigned>(grid), 32 * kSmWarps, sizeof(SmallMSmem), stream>>>(p, y, ldy);
  return cudaGetLastError();
}

}  // namespace w4a4
