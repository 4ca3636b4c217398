// Block-scaled W4A4 GEMM, warp-level tensor-core version (mma.sync, e4m3).
//
// Engine docs "The lean option: ROCmFP4, ROCmI4 and Hadamard Q4_0", section
// "Hadamard-rotated Q4_0: W4A4 prompt processing": int4 weights times int4
// activations on the matrix units, a Q4_0 code q standing for q - 8 (q ^ 8 as a
// signed nibble); section "MoE: W4A4 on the experts": the same kernel on the
// routed expert matmuls (MUL_MAT_ID).
//
//   P[m][n][b] = sum_{j<32} (q_w - 8) q_a           one m16n8k32 MMA per block
//   Y[m][n]   += d_w[n][b] * d_a[m][b] * P[m][n][b]  fp32 fold in registers
//
// GB300 has no integer tcgen05 kind on sm_103a, so the exact integer dot runs
// as fp8: every int4 value v is the e4m3 value v * 2^-9 (see w4a4_device.cuh),
// the 32-term sum comes out of the fp32 accumulator as P * 2^-18 exactly, and
// 2^18 is folded into the weight scale.  The MMA C operand is zero for every
// block, so no rounding ever mixes two blocks before their scales are applied.
//
// CTA tile: 128 activation rows x 128 weight rows, 8 warps as 2 x 4, warp tile
// 64 x 32 (4 x 4 MMAs per block).  Codes and scales are staged by cp.async in a
// 3-deep ring of 4-block stages; code rows are padded to 80 bytes so that the
// fragment loads (word t of rows g = 0..7) hit 32 distinct banks.
#include "w4a4_kernels.cuh"

namespace w4a4 {

namespace {

constexpr int BM = kGemmBM;
constexpr int BN = kGemmBN;
constexpr int KB = 4;               // 32-blocks per stage
constexpr int STAGES = 3;
constexpr int ROWB = KB * 16 + 16;  // padded code row (bytes)
constexpr int THREADS = 256;

struct Stage {
  uint8_t a[BM * ROWB];
  uint8_t w[BN * ROWB];
  float as[BM * KB];      // activation scales
  uint32_t ws[BN * KB];   // weight scale words (raw fp16 pair, then fp32 * 2^18)
};
constexpr size_t kSmemBytes = sizeof(Stage) * STAGES;

enum class Mode { kFold, kPartials };

struct Args {
  const uint8_t* a_codes;
  const float* a_scales;
  const uint8_t* w_codes;
  const uint16_t* w_scales;
  int64_t M, N, K;
  float* y;
  int64_t ldy;
  int32_t* P;
  // routed (MUL_MAT_ID) only
  const int32_t* perm;
  const int32_t* offsets;
  const int32_t* tile_off;
  int E;
  int top_k;
  int act_per_slot;
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool pred) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(pred ? 16 : 0));
}
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem, bool pred) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(s), "l"(gmem), "r"(pred ? 4 : 0));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void mma_e4m3(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};\n"
      : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]), "f"(0.0f));
}

template <Mode MODE, bool ROUTED>
__global__ void __launch_bounds__(THREADS) w4a4_gemm_mma_kernel(Args p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Stage* st = reinterpret_cast<Stage*>(smem_raw);
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int wm = warp >> 2, wn = warp & 3;
  const int64_t B = p.K / 32;
  const int64_t n0 = static_cast<int64_t>(blockIdx.y) * BN;

  // ---- which activation rows this CTA owns
  int64_t m0 = static_cast<int64_t>(blockIdx.x) * BM;
  int rows = 0;  // valid activation rows in this tile
  int64_t pair0 = 0;
  const uint8_t* wc = p.w_codes;
  const uint16_t* wsc = p.w_scales;
  if constexpr (ROUTED) {
    const int mt = blockIdx.x;
    if (mt >= p.tile_off[p.E]) return;
    int lo = 0, hi = p.E - 1;  // last expert with tile_off[e] <= mt
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.tile_off[mid] <= mt) lo = mid; else hi = mid - 1;
    }
    const int e = lo;
    pair0 = p.offsets[e] + static_cast<int64_t>(mt - p.tile_off[e]) * BM;
    {
      const int64_t left = p.offsets[e + 1] - pair0;
      rows = static_cast<int>(left < BM ? left : BM);
    }
    wc += static_cast<int64_t>(e) * p.N * (p.K / 2);
    wsc += static_cast<int64_t>(e) * p.N * B;
  } else {
    {
      const int64_t left = p.M - m0;
      rows = static_cast<int>(left < BM ? left : BM);
    }
  }

  // ---- per-thread load assignment: rows r0, r0 + 64, 16-byte chunk / block `ch`
  const int ch = tid & 3;
  const int r0 = tid >> 2;
  const uint8_t* a_row[2];
  const float* as_row[2];
  bool a_ok[2];
  const uint8_t* w_row[2];
  const uint16_t* ws_row[2];
  int64_t ws_idx[2];
  bool w_ok[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = r0 + 64 * i;
    a_ok[i] = r < rows;
    int64_t arow = 0;
    if (a_ok[i]) {
      if constexpr (ROUTED) {
        const int64_t pr = p.perm[pair0 + r];
        arow = p.act_per_slot ? pr : pr / p.top_k;
      } else {
        arow = m0 + r;
      }
    }
    a_row[i] = p.a_codes + arow * (p.K / 2);
    as_row[i] = p.a_scales + arow * B;
    const int64_t wr = n0 + r;
    w_ok[i] = wr < p.N;
    const int64_t wrc = w_ok[i] ? wr : 0;
    w_row[i] = wc + wrc * (p.K / 2);
    ws_row[i] = wsc;
    ws_idx[i] = wrc * B;
  }

  const int64_t nstages = (B + KB - 1) / KB;
  auto load_stage = [&](int64_t s) {
    Stage& S = st[s % STAGES];
    const int64_t b = s * KB + ch;
    const bool bok = b < B;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = r0 + 64 * i;
      cp_async16(S.a + r * ROWB + ch * 16, a_row[i] + (bok ? b * 16 : 0), a_ok[i] && bok);
      cp_async16(S.w + r * ROWB + ch * 16, w_row[i] + (bok ? b * 16 : 0), w_ok[i] && bok);
      cp_async4(S.as + r * KB + ch, as_row[i] + (bok ? b : 0), a_ok[i] && bok);
      const int64_t hidx = ws_idx[i] + (bok ? b : 0);
      cp_async4(S.ws + r * KB + ch, ws_row[i] + (hidx & ~int64_t(1)), w_ok[i] && bok);
    }
  };

  float acc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[i][j][k] = 0.f;

  const bool warp_active = wm * 64 < rows;  // warps above the tile's last row skip the math

#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < nstages) load_stage(s);
    cp_async_commit();
  }

  for (int64_t s = 0; s < nstages; ++s) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();
    Stage& S = st[s % STAGES];
    // weight scale words -> fp32 * 2^18 (each thread converts the two it loaded)
    {
      const int64_t b = s * KB + ch;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int r = r0 + 64 * i;
        const uint32_t word = S.ws[r * KB + ch];
        const int64_t hidx = ws_idx[i] + (b < B ? b : 0);
        const uint16_t h = static_cast<uint16_t>((hidx & 1) ? (word >> 16) : (word & 0xFFFFu));
        const float f = __half2float(__ushort_as_half(h)) * fp8_unscale();
        S.ws[r * KB + ch] = __float_as_uint(f);
      }
    }
    if (s + STAGES - 1 < nstages) load_stage(s + STAGES - 1);
    cp_async_commit();
    __syncthreads();

    if (warp_active) {
      const float* wsf = reinterpret_cast<const float*>(S.ws);
#pragma unroll 1
      for (int kb = 0; kb < KB; ++kb) {
        const int64_t bglob = s * KB + kb;
        if (bglob >= B) break;
        uint32_t af[4][4], bf[4][2];
        float da[4][2], dw[4][2];
#pragma unroll
        for (int mi = 0; mi < 4; ++mi) {
          const int ra = wm * 64 + mi * 16 + g;
          const uint32_t w0 = *reinterpret_cast<const uint32_t*>(S.a + ra * ROWB + kb * 16 + 4 * t);
          const uint32_t w1 = *reinterpret_cast<const uint32_t*>(S.a + (ra + 8) * ROWB + kb * 16 + 4 * t);
          act_word_to_e4m3(w0, af[mi][0], af[mi][2]);
          act_word_to_e4m3(w1, af[mi][1], af[mi][3]);
          da[mi][0] = S.as[ra * KB + kb];
          da[mi][1] = S.as[(ra + 8) * KB + kb];
        }
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
          const int rw = wn * 32 + ni * 8 + g;
          const uint32_t wv = *reinterpret_cast<const uint32_t*>(S.w + rw * ROWB + kb * 16 + 4 * t);
          q4_0_word_to_e4m3(wv, bf[ni][0], bf[ni][1]);
          const int cw = wn * 32 + ni * 8 + 2 * t;
          dw[ni][0] = wsf[cw * KB + kb];
          dw[ni][1] = wsf[(cw + 1) * KB + kb];
        }
#pragma unroll
        for (int mi = 0; mi < 4; ++mi) {
#pragma unroll
          for (int ni = 0; ni < 4; ++ni) {
            float c[4];
            mma_e4m3(c, af[mi], bf[ni]);
            if constexpr (MODE == Mode::kFold) {
              acc[mi][ni][0] = fmaf(c[0] * dw[ni][0], da[mi][0], acc[mi][ni][0]);
              acc[mi][ni][1] = fmaf(c[1] * dw[ni][1], da[mi][0], acc[mi][ni][1]);
              acc[mi][ni][2] = fmaf(c[2] * dw[ni][0], da[mi][1], acc[mi][ni][2]);
              acc[mi][ni][3] = fmaf(c[3] * dw[ni][1], da[mi][1], acc[mi][ni][3]);
            } else {
              const int ra = wm * 64 + mi * 16 + g;
              const int64_t col = n0 + wn * 32 + ni * 8 + 2 * t;
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int64_t m = m0 + ra + 8 * h;
                if (ra + 8 * h < rows) {
#pragma unroll
                  for (int j = 0; j < 2; ++j) {
                    if (col + j < p.N) {
                      const float v = c[2 * h + j] * fp8_unscale();
                      p.P[(m * p.N + col + j) * B + bglob] = static_cast<int32_t>(v);
                    }
                  }
                }
              }
            }
          }
        }
      }
    }
  }
  cp_async_wait<0>();

  if constexpr (MODE == Mode::kFold) {
    // paired stores need 8-byte aligned rows
    const bool vec2 = ((reinterpret_cast<uintptr_t>(p.y) & 7u) == 0) && ((p.ldy & 1) == 0);
    if (!warp_active) {
      // rows of a partial tile still get written below (zeros are correct only for
      // rows that exist; inactive warps own no existing rows)
      return;
    }
#pragma unroll
    for (int mi = 0; mi < 4; ++mi) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int ra = wm * 64 + mi * 16 + g + 8 * h;
        if (ra >= rows) continue;
        int64_t yrow;
        if constexpr (ROUTED) {
          yrow = p.perm[pair0 + ra];
        } else {
          yrow = m0 + ra;
        }
        float* yr = p.y + yrow * p.ldy;
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
          const int64_t col = n0 + wn * 32 + ni * 8 + 2 * t;
          const float v0 = acc[mi][ni][2 * h], v1 = acc[mi][ni][2 * h + 1];
          if (col + 1 < p.N && vec2) {
            *reinterpret_cast<float2*>(yr + col) = make_float2(v0, v1);
          } else if (col + 1 < p.N) {
            yr[col] = v0;
            yr[col + 1] = v1;
          } else if (col < p.N) {
            yr[col] = v0;
          }
        }
      }
    }
  }
}

template <Mode MODE, bool ROUTED>
cudaError_t launch(const Args& a, dim3 grid, cudaStream_t stream) {
  auto kern = w4a4_gemm_mma_kernel<MODE, ROUTED>;
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  kern<<<grid, THREADS, kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm(const uint8_t* w_codes, const uint16_t* w_scales, int64_t N, const uint8_t* a_codes,
                        const float* a_scales, int64_t M, int64_t K, float* y, int64_t ldy, cudaStream_t stream) {
  Args a{};
  a.a_codes = a_codes; a.a_scales = a_scales; a.w_codes = w_codes; a.w_scales = w_scales;
  a.M = M; a.N = N; a.K = K; a.y = y; a.ldy = ldy;
  const dim3 grid(static_cast<unsigned>((M + BM - 1) / BM), static_cast<unsigned>((N + BN - 1) / BN));
  return launch<Mode::kFold, false>(a, grid, stream);
}

cudaError_t launch_gemm_partials(const uint8_t* w_codes, const uint16_t* w_scales, int64_t N,
                                 const uint8_t* a_codes, const float* a_scales, int64_t M, int64_t K, int32_t* P,
                                 cudaStream_t stream) {
  Args a{};
  a.a_codes = a_codes; a.a_scales = a_scales; a.w_codes = w_codes; a.w_scales = w_scales;
  a.M = M; a.N = N; a.K = K; a.P = P;
  const dim3 grid(static_cast<unsigned>((M + BM - 1) / BM), static_cast<unsigned>((N + BN - 1) / BN));
  return launch<Mode::kPartials, false>(a, grid, stream);
}

cudaError_t launch_gemm_routed(const uint8_t* w_codes, const uint16_t* w_scales, int E, int64_t N,
                               const uint8_t* a_codes, const float* a_scales, int64_t K, int64_t npairs, int top_k,
                               int act_per_slot, float* y, const Routing& r, cudaStream_t stream) {
  Args a{};
  a.a_codes = a_codes; a.a_scales = a_scales; a.w_codes = w_codes; a.w_scales = w_scales;
  a.M = npairs; a.N = N; a.K = K; a.y = y; a.ldy = N;
  a.perm = r.perm; a.offsets = r.offsets; a.tile_off = r.tile_off; a.E = E; a.top_k = top_k;
  a.act_per_slot = act_per_slot;
  const int64_t max_tiles = npairs / BM + E;
  const dim3 grid(static_cast<unsigned>(max_tiles), static_cast<unsigned>((N + BN - 1) / BN));
  return launch<Mode::kFold, true>(a, grid, stream);
}

}  // namespace w4a4
