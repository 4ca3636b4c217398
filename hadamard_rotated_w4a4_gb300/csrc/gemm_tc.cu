// Block-scaled W4A4 GEMM on the 5th-generation tensor cores (tcgen05, TMEM).
//
// Engine docs "The lean option: ROCmFP4, ROCmI4 and Hadamard Q4_0", section
// "Hadamard-rotated Q4_0: W4A4 prompt processing": int4 weights times int4
// activations on the matrix units, weights read as plain Q4_0 (code q stands for
// q - 8); section "MoE: W4A4 on the experts": the same product on the routed
// expert matmuls (MUL_MAT_ID).
//
//   P[n][m][b] = sum_{j<32} (q_w - 8) q_a            exact, on the tensor cores
//   Y[m][n]   += d_w[n][b] * d_a[m][b] * P[n][m][b]   fp32 fold on the CUDA cores
//
// Exact integer dot on fp8 hardware.  sm_103a has no integer tcgen05 kind, but
// every 4-bit value v is exactly the e4m3 value v * 2^-9 (bytes 0x00..0x0F are
// linear, 0x80 adds the sign), so one kind::f8f6f4 MMA with K = 32 yields
// P * 2^-18 in fp32 without rounding; 2^18 is folded into the weight scale.
// Weights enter as signed values q - 8 (a q ^ 8 nibble converted to
// sign-magnitude).  Activations enter as the unsigned offset codes u = a + 8
// (two's complement nibble with bit 3 flipped, no sign logic), and a second MMA
// per block against a constant -8 operand adds -8 * sum_j (q_w - 8), so the
// accumulator holds exactly sum_j (q_w - 8)(u - 8) = P.
//
// Tile: 128 weight rows (MMA M = the 128 TMEM lanes) x up to 256 token columns
// (MMA N), two TMEM accumulator buffers (512 columns) so that the MMA of block
// b + 1 overlaps the fold of block b.  Warp roles (384 threads, 1 CTA per SM):
//   warp 0      producer: cp.async.bulk of each row's packed codes for a stage
//               of 4 blocks into a 3-deep raw ring (mbarrier complete_tx);
//   warp 1      TMEM allocator and MMA issuer (one thread);
//   warps 2-3   converters: unpack int4 -> fp8 into the MMA operand layout
//               (K-major 8-row x 16-byte core matrices), 4 buffers ahead;
//   warps 4-11  workers: load each stage's scales and fold each block's
//               accumulator (tcgen05.ld) into fp32 registers; store Y.
// Warpgroup 0 releases registers (setmaxnreg.dec) to the two worker
// warpgroups (setmaxnreg.inc), which hold 128 fp32 accumulators per thread.
// Every mbarrier wait is bounded (globaltimer); a wait that gives up sets a
// device error word (read by w4a4_check) and the CTA winds down.
#include "w4a4_kernels.cuh"

namespace w4a4 {

// Nonzero once a bounded wait in a GEMM kernel gave up (read and cleared by
// w4a4_check through cudaMemcpyFromSymbol / ToSymbol).
__device__ int g_w4a4_device_error;

namespace {

constexpr int kWorkerWarps = 8;                 // warpgroups 1 and 2: fold
constexpr int kConvWarps = 2;                   // warps 2-3 of warpgroup 0: int4 -> fp8
constexpr int kThreads = 128 + 32 * kWorkerWarps;
constexpr int kRegsLow = 80;    // warpgroup 0 after setmaxnreg.dec
constexpr int kRegsHigh = 208;  // warpgroups 1-2 after setmaxnreg.inc
constexpr int TW = 128;             // weight rows per tile
constexpr int TT = 256;             // token columns per tile (max)
constexpr int KB = 4;               // 32-blocks per raw stage
constexpr int RAW = 3;              // raw stages in flight
constexpr int F8 = 4;               // converted operand buffers
constexpr int RROW = KB * 16 + 16;  // padded raw row: 8 consecutive rows hit distinct banks
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kTimeoutNs = 1000000000ull;  // 1 s

struct __align__(1024) Smem {
  uint8_t wf8[F8][TW * 32];
  uint8_t af8[F8][TT * 32];
  uint8_t cneg[TT * 32];
  uint8_t wraw[RAW][TW * RROW];
  uint8_t araw[RAW][TT * RROW];
  float sda[2][KB][TT];
  float sdw[2][KB][TW];
  uint64_t full_raw[RAW];
  uint64_t empty_raw[RAW];
  uint64_t f8_full[F8];
  uint64_t f8_empty[F8];
  uint64_t tm_full[2];
  uint64_t tm_empty[2];
  uint64_t sc_ready[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  volatile int abort;
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;  // + alignment slack

struct TcArgs {
  const uint8_t* w_codes;
  const uint16_t* w_scales;
  const uint8_t* a_codes;
  const float* a_scales;
  int64_t M;  // dense: token rows; routed: (token, slot) pairs
  int64_t N;  // output features (per expert)
  int64_t K;
  float* y;
  int64_t ldy;
  int32_t* P;
  int tt;  // token tile (multiple of 32, <= TT)
  const int32_t* perm;
  const int32_t* offsets;
  const int32_t* tile_off;
  int E;
  int top_k;
  int act_per_slot;
};

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t su32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t gtime() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
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
// Bounded wait on phase `parity`; false if it (or another role) gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, Smem& S) {
  if (mbar_try(b, parity)) return true;
  const uint64_t t0 = gtime();
  for (;;) {
    if (mbar_try(b, parity)) return true;
    if (S.abort) return false;
    if (gtime() - t0 > kTimeoutNs) {
      S.abort = 1;
      atomicOr(&g_w4a4_device_error, 1);
      return false;
    }
  }
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(su32(dst)),
      "l"(src), "r"(bytes), "r"(su32(bar))
      : "memory");
}
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// K-major operand without swizzle: 8-row x 16-byte core matrices, the two
// 16-byte halves of a 32-byte row 128 bytes apart (LBO), 8-row groups 256 bytes
// apart (SBO); descriptor version 1 (bits 46-47).
__device__ __forceinline__ uint64_t kmajor_desc(const void* smem) {
  const uint32_t a = su32(smem);
  return static_cast<uint64_t>((a >> 4) & 0x3FFFu) | (static_cast<uint64_t>(128 >> 4) << 16) |
         (static_cast<uint64_t>(256 >> 4) << 32) | (static_cast<uint64_t>(1) << 46);
}
// kind::f8f6f4 instruction descriptor: D f32, A and B e4m3, both K-major, M = 128.
__device__ __forceinline__ uint32_t f8_idesc(int n) {
  return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);
}
__device__ __forceinline__ void mma_f8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, int acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
               : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ------------------------------------------------------------------ tiles
struct Tile {
  int64_t n0;     // first weight row of the tile within its expert
  int64_t wbase;  // first weight row in the stacked weight array
  int64_t m0;     // dense: first token row; routed: first pair of the segment
  int rows_w;     // valid weight rows (<= 128)
  int ntok;       // valid token rows (<= tt)
  int nmma;       // MMA N: ntok rounded up to 32
};

__device__ __forceinline__ int64_t num_tiles(const TcArgs& p) {
  const int64_t ntw = (p.N + TW - 1) / TW;
  if (p.tile_off) return static_cast<int64_t>(p.tile_off[p.E]) * ntw;
  return ntw * ((p.M + p.tt - 1) / p.tt);
}

__device__ __forceinline__ Tile decode_tile(const TcArgs& p, int64_t t) {
  Tile T;
  const int64_t ntw = (p.N + TW - 1) / TW;
  int64_t wt;
  if (p.tile_off) {
    const int64_t mt = t / ntw;
    wt = t - mt * ntw;
    int lo = 0, hi = p.E - 1;  // last expert whose first tile is <= mt
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.tile_off[mid] <= mt) lo = mid; else hi = mid - 1;
    }
    T.m0 = p.offsets[lo] + (mt - p.tile_off[lo]) * p.tt;
    const int64_t left = p.offsets[lo + 1] - T.m0;
    T.ntok = static_cast<int>(left < p.tt ? left : p.tt);
    T.wbase = static_cast<int64_t>(lo) * p.N;
  } else {
    const int64_t ntt = (p.M + p.tt - 1) / p.tt;
    wt = t / ntt;
    const int64_t tt = t - wt * ntt;
    T.m0 = tt * p.tt;
    const int64_t left = p.M - T.m0;
    T.ntok = static_cast<int>(left < p.tt ? left : p.tt);
    T.wbase = 0;
  }
  T.n0 = wt * TW;
  const int64_t lw = p.N - T.n0;
  T.rows_w = static_cast<int>(lw < TW ? lw : TW);
  T.nmma = (T.ntok + 31) & ~31;
  return T;
}

__device__ __forceinline__ int64_t act_row(const TcArgs& p, const Tile& T, int r) {
  if (p.tile_off) {
    const int64_t pr = p.perm[T.m0 + r];
    return p.act_per_slot ? pr : pr / p.top_k;
  }
  return T.m0 + r;
}
__device__ __forceinline__ int64_t out_row(const TcArgs& p, const Tile& T, int r) {
  return p.tile_off ? static_cast<int64_t>(p.perm[T.m0 + r]) : T.m0 + r;
}

// ------------------------------------------------------------------ roles
__device__ void producer_loop(const TcArgs& p, Smem& S, uint32_t& gstage) {
  const int lane = threadIdx.x & 31;
  const int64_t B = p.K / 32;
  const int64_t nst = (B + KB - 1) / KB;
  const int64_t ntiles = num_tiles(p);
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const Tile T = decode_tile(p, t);
    const uint8_t* wrow[TW / 32];
    const uint8_t* arow[TT / 32];
#pragma unroll
    for (int i = 0; i < TW / 32; ++i) {
      const int r = lane + 32 * i;
      wrow[i] = p.w_codes + (T.wbase + T.n0 + (r < T.rows_w ? r : 0)) * (p.K / 2);
    }
#pragma unroll
    for (int i = 0; i < TT / 32; ++i) {
      const int r = lane + 32 * i;
      arow[i] = p.a_codes + act_row(p, T, r < T.ntok ? r : 0) * (p.K / 2);
    }
    for (int64_t s = 0; s < nst; ++s) {
      const int slot = gstage % RAW;
      if (!mbar_wait(&S.empty_raw[slot], ((gstage / RAW) & 1) ^ 1, S)) return;
      const int64_t kb0 = s * KB;
      const uint32_t nbk = static_cast<uint32_t>(B - kb0 < KB ? B - kb0 : KB);
      const uint32_t rb = nbk * 16;
      if (lane == 0) mbar_expect_tx(&S.full_raw[slot], rb * static_cast<uint32_t>(T.rows_w + T.ntok));
      __syncwarp();
#pragma unroll
      for (int i = 0; i < TW / 32; ++i) {
        const int r = lane + 32 * i;
        if (r < T.rows_w) bulk_g2s(S.wraw[slot] + r * RROW, wrow[i] + kb0 * 16, rb, &S.full_raw[slot]);
      }
#pragma unroll
      for (int i = 0; i < TT / 32; ++i) {
        const int r = lane + 32 * i;
        if (r < T.ntok) bulk_g2s(S.araw[slot] + r * RROW, arow[i] + kb0 * 16, rb, &S.full_raw[slot]);
      }
      ++gstage;
    }
  }
}

__device__ void producer(const TcArgs& p, Smem& S) {
  uint32_t gstage = 0;  // stages whose copies were issued
  producer_loop(p, S, gstage);
  // Drain: the last RAW stages' copies must have landed before the CTA exits
  // (normally the workers have already consumed them and this returns at once).
  const uint32_t first = gstage > RAW ? gstage - RAW : 0;
  for (uint32_t g = first; g < gstage; ++g) {
    const uint64_t t0 = gtime();
    while (!mbar_try(&S.full_raw[g % RAW], (g / RAW) & 1) && gtime() - t0 < kTimeoutNs) {
    }
  }
}

__device__ void mma_issuer(const TcArgs& p, Smem& S, uint32_t tmem) {
  const int64_t B = p.K / 32;
  const int64_t ntiles = num_tiles(p);
  const uint64_t cdesc = kmajor_desc(S.cneg);
  uint32_t gblk = 0;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const Tile T = decode_tile(p, t);
    const uint32_t idesc = f8_idesc(T.nmma);
    for (int64_t b = 0; b < B; ++b, ++gblk) {
      const int f = gblk % F8;
      const int tb = gblk & 1;
      if (!mbar_wait(&S.f8_full[f], (gblk / F8) & 1, S)) goto done;
      if (!mbar_wait(&S.tm_empty[tb], ((gblk >> 1) & 1) ^ 1, S)) goto done;
      tc_fence_after();
      {
        const uint32_t d = tmem + static_cast<uint32_t>(tb * TT);
        const uint64_t wdesc = kmajor_desc(S.wf8[f]);
        mma_f8(d, wdesc, kmajor_desc(S.af8[f]), idesc, 0);
        mma_f8(d, wdesc, cdesc, idesc, 1);
      }
      mma_commit(&S.tm_full[tb]);
      mma_commit(&S.f8_empty[f]);
    }
  }
done:
  // wait (bounded) until every issued MMA has finished before TMEM is released
  mma_commit(&S.mma_done);
  {
    const uint64_t t0 = gtime();
    while (!mbar_try(&S.mma_done, 0) && gtime() - t0 < kTimeoutNs) {
    }
  }
}

__device__ void converters(const TcArgs& p, Smem& S) {
  const int ct = threadIdx.x - 64;  // 0..63
  const int lane = threadIdx.x & 31;
  const int64_t B = p.K / 32;
  const int64_t nst = (B + KB - 1) / KB;
  const int64_t ntiles = num_tiles(p);
  uint32_t gstage = 0, gconv = 0;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const Tile T = decode_tile(p, t);
    for (int64_t b = 0; b < B; ++b) {
      const int64_t s = b / KB;
      const int kb = static_cast<int>(b - s * KB);
      const uint32_t gs = gstage + static_cast<uint32_t>(s);
      const int slot = gs % RAW;
      if (kb == 0 && !mbar_wait(&S.full_raw[slot], (gs / RAW) & 1, S)) return;
      const int f = gconv % F8;
      if (!mbar_wait(&S.f8_empty[f], ((gconv / F8) & 1) ^ 1, S)) return;
      // weights: rows ct and ct + 64, signed q - 8
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int r = ct + 64 * i;
        if (r < T.rows_w) {
          const uint4 raw = *reinterpret_cast<const uint4*>(S.wraw[slot] + r * RROW + kb * 16);
          uint32_t l0, h0, l1, h1, l2, h2, l3, h3;
          q4_0_word_to_e4m3(raw.x, l0, h0);
          q4_0_word_to_e4m3(raw.y, l1, h1);
          q4_0_word_to_e4m3(raw.z, l2, h2);
          q4_0_word_to_e4m3(raw.w, l3, h3);
          uint8_t* dst = S.wf8[f] + (r >> 3) * 256 + (r & 7) * 16;
          *reinterpret_cast<uint4*>(dst) = make_uint4(l0, l1, l2, l3);
          *reinterpret_cast<uint4*>(dst + 128) = make_uint4(h0, h1, h2, h3);
        }
      }
      // activations: rows ct + 64 i; offset codes u = a + 8 are the e4m3 bytes themselves
#pragma unroll
      for (int i = 0; i < TT / 64; ++i) {
        const int r = ct + 64 * i;
        if (r < T.nmma) {
          uint4 raw = make_uint4(0u, 0u, 0u, 0u);
          if (r < T.ntok) raw = *reinterpret_cast<const uint4*>(S.araw[slot] + r * RROW + kb * 16);
          const uint32_t x0 = raw.x ^ 0x88888888u, x1 = raw.y ^ 0x88888888u;
          const uint32_t x2 = raw.z ^ 0x88888888u, x3 = raw.w ^ 0x88888888u;
          uint8_t* dst = S.af8[f] + (r >> 3) * 256 + (r & 7) * 16;
          *reinterpret_cast<uint4*>(dst) =
              make_uint4(x0 & 0x0F0F0F0Fu, x1 & 0x0F0F0F0Fu, x2 & 0x0F0F0F0Fu, x3 & 0x0F0F0F0Fu);
          *reinterpret_cast<uint4*>(dst + 128) = make_uint4((x0 >> 4) & 0x0F0F0F0Fu, (x1 >> 4) & 0x0F0F0F0Fu,
                                                            (x2 >> 4) & 0x0F0F0F0Fu, (x3 >> 4) & 0x0F0F0F0Fu);
        }
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&S.f8_full[f]);
        if (kb == KB - 1 || b == B - 1) mbar_arrive(&S.empty_raw[slot]);
      }
      ++gconv;
    }
    gstage += static_cast<uint32_t>(nst);
  }
}

template <bool PARTIALS>
__device__ void workers(const TcArgs& p, Smem& S, uint32_t tmem) {
  const int wt = threadIdx.x - 128;  // 0..255
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;  // 4..11
  const int q = warp & 3;             // TMEM lane quarter this warp may access
  const int h = (warp - 4) >> 2;      // column half: chunks h, h+2, h+4, h+6
  const int n_in = 32 * q + lane;     // this thread's weight row within the tile
  const int B = static_cast<int>(p.K / 32);
  const int nst = (B + KB - 1) / KB;
  const int64_t ntiles = num_tiles(p);
  uint32_t gfold = 0, gsc = 0;

  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const Tile T = decode_tile(p, t);
    const int nchunks = T.nmma / 32;
    // scale sources of this thread: activation row wt, weight row wt (wt < 128)
    const bool a_ok = wt < T.ntok;
    const bool w_ok = wt < T.rows_w;
    const float* as_row = p.a_scales + (a_ok ? act_row(p, T, wt) : 0) * B;
    const uint16_t* ws_row = p.w_scales + (T.wbase + T.n0 + (w_ok ? wt : 0)) * B;
    float da_r[KB], dw_r[KB];
    auto load_scales = [&](int s) {
#pragma unroll
      for (int k = 0; k < KB; ++k) {
        const int b = s * KB + k;
        const bool bok = b < B;
        da_r[k] = (a_ok && bok) ? __ldg(as_row + b) : 0.f;
        dw_r[k] = (w_ok && bok) ? __half2float(__ushort_as_half(__ldg(ws_row + b))) * fp8_unscale() : 0.f;
      }
    };
    // publish the registers' scales for one stage and wait until every worker warp has
    auto publish_scales = [&]() -> bool {
      const int slot = gsc & 1;
#pragma unroll
      for (int k = 0; k < KB; ++k) {
        S.sda[slot][k][wt] = da_r[k];
        if (wt < TW) S.sdw[slot][k][wt] = dw_r[k];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.sc_ready[slot]);
      const bool ok = mbar_wait(&S.sc_ready[slot], (gsc >> 1) & 1, S);
      ++gsc;
      return ok;
    };
    float acc[4][32];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[i][j] = 0.f;

    load_scales(0);
    if (!publish_scales()) return;
    if (nst > 1) load_scales(1);

    for (int b = 0; b < B; ++b) {
      const int s = b / KB;
      const int kb = b - s * KB;
      if (kb == 0 && b > 0) {
        if (!publish_scales()) return;
        if (s + 1 < nst) load_scales(s + 1);
      }
      // ---- fold block b
      const int tb = gfold & 1;
      if (!mbar_wait(&S.tm_full[tb], (gfold >> 1) & 1, S)) return;
      tc_fence_after();
      const int slot = (gsc - 1) & 1;
      const float dw = S.sdw[slot][kb][n_in];
      const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(tb * TT);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = h + 2 * i;
        if (c < nchunks) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float v[16];
            tmem_ld16(tbase + static_cast<uint32_t>(c * 32 + 16 * half), v);
            if constexpr (PARTIALS) {
              const int64_t n = T.n0 + n_in;
#pragma unroll 1
              for (int j = 0; j < 16; ++j) {
                const int col = c * 32 + 16 * half + j;
                if (col < T.ntok && n_in < T.rows_w) {
                  const int64_t m = T.m0 + col;
                  p.P[(m * p.N + n) * B + b] = static_cast<int32_t>(v[j] * fp8_unscale());
                }
              }
            } else {
              const float4* da4 = reinterpret_cast<const float4*>(&S.sda[slot][kb][c * 32 + 16 * half]);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float4 d = da4[j];
                const int o = 16 * half + 4 * j;
                acc[i][o + 0] = fmaf(v[4 * j + 0] * dw, d.x, acc[i][o + 0]);
                acc[i][o + 1] = fmaf(v[4 * j + 1] * dw, d.y, acc[i][o + 1]);
                acc[i][o + 2] = fmaf(v[4 * j + 2] * dw, d.z, acc[i][o + 2]);
                acc[i][o + 3] = fmaf(v[4 * j + 3] * dw, d.w, acc[i][o + 3]);
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.tm_empty[tb]);
      ++gfold;
    }

    if constexpr (!PARTIALS) {
      if (n_in < T.rows_w) {
        const int64_t n = T.n0 + n_in;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = h + 2 * i;
          if (c < nchunks) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int col = c * 32 + j;
              if (col < T.ntok) p.y[out_row(p, T, col) * p.ldy + n] = acc[i][j];
            }
          }
        }
      }
    }
  }
}

template <bool PARTIALS>
__global__ void __launch_bounds__(kThreads, 1) w4a4_gemm_tc_kernel(const TcArgs p) {
  extern __shared__ uint8_t smem_dyn[];
  Smem& S = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    for (int i = 0; i < RAW; ++i) {
      mbar_init(&S.full_raw[i], 1);
      mbar_init(&S.empty_raw[i], kConvWarps);
    }
    for (int i = 0; i < F8; ++i) {
      mbar_init(&S.f8_full[i], kConvWarps);
      mbar_init(&S.f8_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.tm_full[i], 1);
      mbar_init(&S.tm_empty[i], kWorkerWarps);
      mbar_init(&S.sc_ready[i], kWorkerWarps);
    }
    mbar_init(&S.mma_done, 1);
    S.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int i = threadIdx.x; i < TT * 32 / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(S.cneg)[i] = 0x88888888u;  // e4m3 -8 * 2^-9
  fence_async_smem();
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&S.tmem_base)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
    if (warp == 0) {
      producer(p, S);
    } else if (warp == 1) {
      if ((threadIdx.x & 31) == 0) mma_issuer(p, S, tmem);
      __syncwarp();
    } else {
      converters(p, S);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
    workers<PARTIALS>(p, S, tmem);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

template <bool PARTIALS>
cudaError_t launch_tc(const TcArgs& a, int64_t max_tiles, cudaStream_t stream) {
  auto kern = w4a4_gemm_tc_kernel<PARTIALS>;
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  // setmaxnreg.inc waits until the block's launch registers cover the split:
  // refuse to launch a build whose register count would make it wait forever.
  static int regs_ok[64] = {};
  if (dev >= 0 && dev < 64 && regs_ok[dev] == 0) {
    cudaFuncAttributes fa{};
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    regs_ok[dev] = (fa.numRegs * kThreads >= 128 * kRegsLow + 256 * kRegsHigh) ? 1 : -1;
  }
  if (dev >= 0 && dev < 64 && regs_ok[dev] < 0) return cudaErrorInvalidConfiguration;
  int64_t grid = max_tiles < num_sms() ? max_tiles : num_sms();
  if (grid < 1) grid = 1;
  kern<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}

int token_tile(int64_t M) {
  const int64_t r = (M + 31) & ~int64_t(31);
  return static_cast<int>(r < TT ? r : TT);
}

}  // namespace

cudaError_t launch_gemm_tc(const uint8_t* w_codes, const uint16_t* w_scales, int64_t N, const uint8_t* a_codes,
                           const float* a_scales, int64_t M, int64_t K, float* y, int64_t ldy, int32_t* P,
                           cudaStream_t stream) {
  TcArgs a{};
  a.w_codes = w_codes; a.w_scales = w_scales; a.a_codes = a_codes; a.a_scales = a_scales;
  a.M = M; a.N = N; a.K = K; a.y = y; a.ldy = ldy; a.P = P;
  a.tt = token_tile(M);
  const int64_t tiles = ((N + TW - 1) / TW) * ((M + a.tt - 1) / a.tt);
  return P ? launch_tc<true>(a, tiles, stream) : launch_tc<false>(a, tiles, stream);
}

cudaError_t launch_gemm_tc_routed(const uint8_t* w_codes, const uint16_t* w_scales, int E, int64_t N,
                                  const uint8_t* a_codes, const float* a_scales, int64_t K, int64_t npairs,
                                  int top_k, int act_per_slot, int tile_tokens, float* y, const Routing& r,
                                  cudaStream_t stream) {
  TcArgs a{};
  a.w_codes = w_codes; a.w_scales = w_scales; a.a_codes = a_codes; a.a_scales = a_scales;
  a.M = npairs; a.N = N; a.K = K; a.y = y; a.ldy = N;
  a.tt = tile_tokens;
  a.perm = r.perm; a.offsets = r.offsets; a.tile_off = r.tile_off; a.E = E; a.top_k = top_k;
  a.act_per_slot = act_per_slot;
  const int64_t max_tiles = (npairs / tile_tokens + E) * ((N + TW - 1) / TW);
  return launch_tc<false>(a, max_tiles, stream);
}

cudaError_t read_and_clear_device_error(int* value) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_w4a4_device_error, sizeof(int));
  if (e != cudaSuccess) return e;
  *value = v;
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_w4a4_device_error, &zero, sizeof(int));
  }
  return e;
}

}  // namespace w4a4
