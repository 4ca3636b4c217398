// Block-scaled W4A4 GEMM on the 5th-generation tensor cores (tcgen05, TMEM, TMA),
// the instance that converts both operands' codes in the kernel: the dense
// product without the expanded activation operand, the exact integer partials,
// and the two other routes (the exact path's int8 activations, the rotate-only
// route's bf16 activations).  The dense product with the expanded activation
// operand and the routed product run in the super-tile kernel (gemm_grp.cu).
//
// Engine docs "The lean option: ROCmFP4, ROCmI4 and Hadamard Q4_0", section
// "Hadamard-rotated Q4_0: W4A4 prompt processing": int4 weights times int4
// activations on the matrix units, weights read as plain Q4_0 (code q stands for
// q - 8).
//
//   P[n][m][b] = sum_{j<32} (q_w - 8) q_a            exact, on the tensor cores
//   Y[m][n]   += d_w[n][b] * d_a[m][b] * P[n][m][b]   fp32 fold on the CUDA cores
//
// Exact integer dot on fp8 hardware.  sm_103a has no integer tcgen05 kind, but
// every 4-bit value v is exactly the e4m3 value v * 2^-9 (bytes 0x00..0x0F are
// linear, 0x80 adds the sign), so one kind::f8f6f4 MMA with K = 32 gives a
// 32-term sum of exact products in fp32, again exact (|sum| <= 3360 * 2^-18).
// Weights enter as signed values q - 8 (the q ^ 8 nibble in sign-magnitude);
// activations as their unsigned offset codes u = a + 8 (a two's complement
// nibble with bit 3 flipped: no sign logic).  The MMA therefore yields
// D = P + 8 S_w with S_w = sum_j (q_w - 8) (stored with the weights), and the
// fold removes 8 S_w inside its first fused multiply-add:
//   t = fma(D * 2^-18, d_w * 2^18, -d_w * 8 S_w) = round(d_w * P)
// -- exact operands (d_w * 8 S_w has at most 20 significant bits), one rounding,
// the same value as multiplying the exact P by d_w -- then acc = fma(t, d_a, acc).
//
// Tile: 128 weight rows (MMA M = the 128 TMEM lanes) x up to 256 token columns
// (MMA N), two TMEM accumulator buffers (512 columns) so that the MMA of block
// b + 1 overlaps the fold of block b.  Warp roles (384 threads, 1 CTA per SM):
//   warp 0      producer: two 2D TMA loads per stage of 4 blocks (the weight and
//               activation code tiles, 64 bytes of each row) into a 3-deep ring;
//   warp 1      TMEM allocator and MMA issuer (one thread, one MMA per block);
//   warps 2-3   converters: unpack a stage's int4 codes into four fp8 operand
//               buffers (K-major 8-row x 16-byte core matrices);
//   warps 4-11  workers: each stage's scales, the fold of each block's
//               accumulator (tcgen05.ld) into 128 fp32 registers per thread, Y.
// Warpgroup 0 releases registers (setmaxnreg.dec) to the two worker warpgroups
// (setmaxnreg.inc).  Every mbarrier wait is bounded (globaltimer); a wait that
// gives up sets a device error word (read by w4a4_check) and the CTA winds down.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>


#include <cuda_bf16.h>

#include "tc_ptx.cuh"
#include "w4a4_kernels.cuh"

namespace w4a4 {

// Nonzero once a bounded wait in a GEMM kernel gave up (read and cleared by
// w4a4_check through cudaMemcpyFromSymbol / ToSymbol).
__device__ int g_w4a4_device_error;

namespace {

constexpr int kWorkerWarps = 8;  // warps 4-11, warpgroups 1-2
constexpr int TW = 128;         // weight rows per tile
// The token tile is a template parameter TTM (256 or 128 token columns).  A
// tile of TTM columns has 512 / TTM accumulator buffers in TMEM, and each worker
// thread holds TTM / 2 accumulators (chunks h + 2i of 32 columns, i < TTM / 64).
constexpr int KB = 4;           // 32-blocks per stage (64 code bytes per row)
static_assert(KB == 4, "the vector scale loads take 4 blocks per stage");
#ifndef W4A4_RAW_STAGES
#define W4A4_RAW_STAGES 3
#endif
#ifndef W4A4_F8_BUFFERS
#define W4A4_F8_BUFFERS 8
#endif
constexpr int RAW = W4A4_RAW_STAGES;  // stages of raw codes in flight
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kTimeoutNs = 1000000000ull;  // 1 s
#ifndef W4A4_WAIT_HINT_NS
#define W4A4_WAIT_HINT_NS 0
#endif
// Suspend-time hint of the mbarrier waits; 0 = poll without suspending, which
// measured about 2% faster than a 20 us hint on the dense workloads.
constexpr uint32_t kWaitHintNs = W4A4_WAIT_HINT_NS;


// Warp roles by token tile.  Warp 0 produces (TMA), warp 1 issues the MMAs,
// warps 4-11 fold.  The 256-column instance has two converter warps (2-3) and
// 384 threads; the 128-column instance, whose workers need fewer registers,
// adds warpgroup 3 as four more converter warps (512 threads) and a third fp8
// stage.  Registers after setmaxnreg: 128 x 56 + 256 x 224 = 168 x 384 (the
// workers' 224 leave the fold loop without spills), and 256 x 72 + 256 x 184 =
// 128 x 512.
// AB: activation code width.  4 = the W4A4 product (int4 activations, e4m3
// operands, one kind::f8f6f4 MMA per block); 8 = the exact path (int8
// activations, f16 operands, two kind::f16 MMAs of K = 16 per block; int8 and
// int4 values are exact in f16 and so are the 32-term block sums in fp32);
// 16 = the rotate-only route (bf16 activations that were not quantised, bf16
// weight operands q - 8, two kind::f16 MMAs per block with the bf16 format;
// the block sums round in the tensor core's fp32 accumulation, d_a = 1).
// WEXP: the weights come pre-expanded (the e4m3 bytes of q - 8, loaded by a 4D
// TMA straight into the K-major operand layout) and the MMA reads them from the
// raw stage; the converters then handle only the activations.
// AEXP (with WEXP, W4A4 only): the activations come pre-expanded as well (the
// offset codes a + 8 as e4m3 bytes, same 4D load); nothing is converted and the
// converter warps only publish the per-stage scales.
template <int TTM, int AB = 4, bool WEXP = false, bool AEXP = false>
struct __align__(128) Smem {
  static_assert(!AEXP || (WEXP && AB == 4), "expanded activations go with expanded weights, W4A4 only");
  static constexpr int TT = TTM;
  static constexpr int ABITS = AB;
  static constexpr bool WX = WEXP;
  static constexpr bool AX = AEXP;
  static constexpr int WROW = KB * (WEXP ? 32 : 16);  // raw weight bytes per row and stage
  static constexpr int ARAW_ROW = AEXP ? KB * 32 : KB * 4 * AB;  // raw activation bytes per row and stage
  static constexpr int OPB = AB == 4 ? 1 : 2;   // operand bytes per element: e4m3 or f16
  static constexpr int WOP = TW * 32 * OPB + 32;   // operand buffer strides, padded by 32 bytes so that the
  static constexpr int AOP = TTM * 32 * OPB + 32;  // converters' stores to 4 buffers hit distinct banks
  static constexpr int NBUF = 512 / TTM;  // TMEM accumulator buffers
  static constexpr int CONV = TTM == 256 ? 2 : 6;                   // converter warps
  static constexpr int THREADS = TTM == 256 ? 384 : 512;
  // (in the expanded-operand instance the converter warps' scale publishing
  // spills a little at 56; it has stages of slack, while the workers' fold runs
  // 2-4% faster at 224 than at 208 -- and 40 / 232 spills in the MMA issuer)
  static constexpr int REGS_LOW = TTM == 256 ? 56 : 72;       // warpgroups 0 and 3
  static constexpr int REGS_HIGH = TTM == 256 ? 224 : 184;    // warpgroups 1-2
  static constexpr int F8 = AB == 16 ? 4 : AB == 8 ? 6 : (TTM == 256 ? W4A4_F8_BUFFERS : 12);  // operand buffers
  // Who writes the per-stage scale slots.  The 128-column instance has converter
  // warps to spare and lets them do it: stage s's scales go to slot s % 4 while
  // stage s is converted, after the converters waited for the MMA to release
  // stage s - F8/4 >= s - 3's operand buffers; those MMAs needed the workers to
  // release every block before them by NBUF = 4 blocks, so the workers are done
  // with stage s - 4, the slot's previous user.  With expanded activations the
  // converters publish stage s into slot s % (RAW + 1) once stage s's codes have
  // landed: the producer refilled that raw slot only after the MMA of the last
  // block of stage s - RAW completed, and that MMA (NBUF = 2) waited for every
  // worker to release block 4(s - RAW) + 1, past the slot's previous user, stage
  // s - RAW - 1.  In the 256-column instance the
  // workers publish stage s + 1's scales during block kb = 2 of stage s into slot
  // (s + 1) % 3, last read by stage s - 2; that block's MMA needed every warp to
  // release block 4s + 2 - NBUF = 4s, past stage s - 2.
  static constexpr bool CONV_SCALES = TTM == 128 || AEXP;
  static constexpr int NSC = AEXP ? RAW + 1 : CONV_SCALES ? 4 : 3;
  uint8_t wraw[RAW][TW * WROW];  // TMA box: 128 rows x 64 code bytes, or (WEXP) the operand layout of 4 blocks
  uint8_t araw[RAW][TTM * ARAW_ROW];  // TMA box: tt rows x 64 (int4) or 128 (int8) bytes
  uint8_t wf8[WEXP ? 1 : F8][WOP];
  uint8_t af8[AEXP ? 1 : F8][AOP];
  float sda[NSC][KB][TTM];              // d_a per stage, block-major
  float sdw[NSC][KB][TW];              // d_w * 2^18
  float scorr[NSC][KB][TW];            // -d_w * 8 S_w (exact)
  uint64_t full_raw[RAW];
  uint64_t empty_raw[RAW];
  uint64_t f8_full[F8];
  uint64_t f8_empty[F8];   // the MMA has read the operand buffer
  uint64_t tm_full[NBUF];
  uint64_t tm_empty[NBUF];
  uint64_t sc_ready[NSC];
  uint64_t tile_done;      // every worker warp has finished its previous tile
  uint64_t mma_done;
  uint32_t tmem_base;
  volatile int abort;
};
static_assert(sizeof(Smem<256>) <= 227 * 1024, "shared memory per CTA is at most 227 KB");
static_assert(sizeof(Smem<128>) <= 227 * 1024, "shared memory per CTA is at most 227 KB");
static_assert(sizeof(Smem<128, 8>) <= 227 * 1024, "shared memory per CTA is at most 227 KB");
static_assert(sizeof(Smem<128, 16>) <= 227 * 1024, "shared memory per CTA is at most 227 KB");
static_assert(sizeof(Smem<256, 4, true>) <= 227 * 1024, "shared memory per CTA is at most 227 KB");
static_assert(sizeof(Smem<128, 4, true>) <= 227 * 1024, "shared memory per CTA is at most 227 KB");
static_assert(sizeof(Smem<256, 4, true, true>) <= 227 * 1024, "shared memory per CTA is at most 227 KB");

struct TcArgs {
  const uint16_t* w_scales;
  const int16_t* w_sums;  // per weight row and block: S_w = sum_j (q_w - 8)
  const float* a_scales;  // [M][B]
  int64_t M;              // token rows
  int64_t N;              // output features (per expert)
  int64_t K;
  float* y;
  int64_t ldy;
  int32_t* P;
  int tt;                 // token tile (multiple of 32, <= the kernel's TTM): the A box height
  // Stream-K schedule (dense product only): the tiles' K stages form one list of
  // sk_units units, cut into gridDim.x equal contiguous ranges.  0 = each CTA
  // takes whole tiles blockIdx.x, blockIdx.x + gridDim.x, ...
  int64_t sk_units;
  uint32_t* sk_count;            // [tiles][8 worker warps] arrivals; zero between launches
  float4* sk_part;               // [2 * gridDim.x][8 warps][32][32 lanes] fp32 partials
};

// ------------------------------------------------------------------ bounded waits
// Bounded wait on phase `parity`; false if it (or another role) gave up.
template <class SM>
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, SM& S) {
  if (mbar_try(b, parity)) return true;
  const uint64_t t0 = gtime();
  for (;;) {
    if (kWaitHintNs ? mbar_try_sleep(b, parity, kWaitHintNs) : mbar_try(b, parity)) return true;
    if (S.abort) return false;
    if (gtime() - t0 > kTimeoutNs) {
      S.abort = 1;
      atomicOr(&g_w4a4_device_error, 1);
      return false;
    }
  }
}
// Bounded spinning wait for the MMA issuer, whose handoffs are on the critical
// path: non-blocking tests, with the abort flag and the time bound checked every
// 64 polls (about 1.5% faster end to end than the blocking wait).
template <class SM>
__device__ __forceinline__ bool mbar_spin(uint64_t* b, uint32_t parity, SM& S) {
  if (mbar_test(b, parity)) return true;
  const uint64_t t0 = gtime();
  for (uint32_t n = 1;; ++n) {
    if (mbar_test(b, parity)) return true;
    if ((n & 63) == 0) {
      if (S.abort) return false;
      if (gtime() - t0 > kTimeoutNs) {
        S.abort = 1;
        atomicOr(&g_w4a4_device_error, 1);
        return false;
      }
    }
  }
}
// ------------------------------------------------------------------ tiles
struct Tile {
  int64_t n0;     // first weight row of the tile within its expert
  int64_t wrow0;  // first weight row in the (stacked) weight tensor
  int64_t m0;     // first token row
  int rows_w;     // valid weight rows (<= 128)
  int ntok;       // valid token rows (<= tt)
  int nmma;       // MMA N: ntok rounded up to 32
};

__device__ __forceinline__ int64_t num_tiles(const TcArgs& p) {
  const int64_t ntw = (p.N + TW - 1) / TW;
  return ntw * ((p.M + p.tt - 1) / p.tt);
}

// Weight-tile major, so that consecutive CTAs share a weight tile in L2.
__device__ __forceinline__ Tile decode_tile(const TcArgs& p, int64_t t) {
  Tile T;
  const int64_t ntt = (p.M + p.tt - 1) / p.tt;
  const int64_t wt = t / ntt;
  const int64_t tt = t - wt * ntt;
  T.m0 = tt * p.tt;
  const int64_t left = p.M - T.m0;
  T.ntok = static_cast<int>(left < p.tt ? left : p.tt);
  T.n0 = wt * TW;
  T.wrow0 = T.n0;
  const int64_t lw = p.N - T.n0;
  T.rows_w = static_cast<int>(lw < TW ? lw : TW);
  T.nmma = (T.ntok + 31) & ~31;
  return T;
}

// ------------------------------------------------------------------ schedule
// A segment: stages [s0, s1) of tile t; `first`: the CTA's first segment.
struct Seg {
  int64_t t;
  int s0, s1;
  bool first;
};
// The iteration state is one position (a unit, or a tile); the CTA's range is
// recomputed from blockIdx at each step, to keep registers free in the workers.
struct SegIter {
  int64_t next;
};
__device__ __forceinline__ int64_t sk_begin(const TcArgs& p, int64_t c) { return c * p.sk_units / gridDim.x; }
__device__ __forceinline__ SegIter seg_iter(const TcArgs& p) {
  SegIter it;
  it.next = p.sk_units ? sk_begin(p, blockIdx.x) : static_cast<int64_t>(blockIdx.x);
  return it;
}
__device__ __forceinline__ bool seg_next(const TcArgs& p, int nst, SegIter& it, Seg& g) {
  if (p.sk_units) {
    const int64_t start = sk_begin(p, blockIdx.x), end = sk_begin(p, blockIdx.x + 1);
    if (it.next >= end) return false;
    g.first = it.next == start;
    g.t = it.next / nst;
    g.s0 = static_cast<int>(it.next - g.t * nst);
    const int64_t left = end - it.next;
    g.s1 = (nst - g.s0 <= left) ? nst : g.s0 + static_cast<int>(left);
    it.next += g.s1 - g.s0;
  } else {
    if (it.next >= num_tiles(p)) return false;
    g.first = it.next == blockIdx.x;
    g.t = it.next;
    g.s0 = 0;
    g.s1 = nst;
    it.next += gridDim.x;
  }
  return true;
}
// The CTA whose unit range holds unit u (ranges are [c U / G, (c + 1) U / G)).
__device__ __forceinline__ int64_t sk_cta_of_unit(const TcArgs& p, int64_t u) {
  const int64_t G = gridDim.x;
  int64_t c = u * G / p.sk_units;
  if (c >= G) c = G - 1;
  for (int i = 0; i < 4 && c > 0 && sk_begin(p, c) > u; ++i) --c;
  for (int i = 0; i < 4 && c + 1 < G && sk_begin(p, c + 1) <= u; ++i) ++c;
  return c;
}
// One arrival on a (tile, warp) ticket: true for the last of `nparts`, which
// also puts the ticket back to zero (no other arrival for it follows in this
// launch), so the workspace needs no clearing between launches, graph replays
// included.
__device__ __forceinline__ bool sk_ticket(uint32_t* ctr, uint32_t nparts) {
  const uint32_t before = atomicAdd(ctr, 1u);
  if (before + 1 != nparts) return false;
  atomicExch(ctr, 0u);
  return true;
}
// A tile cut by the stream-K ranges: each of its worker warps stores its fp32
// partial accumulators (sk_store, in the worker), then takes a ticket.  The warp
// that arrives last for its (tile, warp) region sums every contributor's partial
// in CTA order -- the same order whichever CTA comes last, so the result does not
// depend on timing -- and writes those outputs.  No CTA waits for another.
__device__ __forceinline__ float4* sk_slot(const TcArgs& p, int64_t cta, bool first, int w, int lane) {
  return p.sk_part + ((2 * cta + (first ? 0 : 1)) * 8 + w) * 1024 + lane;
}
__device__ __forceinline__ bool sk_arrive(const TcArgs& p, int64_t t, int nst, int w, int lane) {
  __threadfence();
  __syncwarp();
  const int64_t u_lo = t * nst;
  const int64_t nparts = sk_cta_of_unit(p, u_lo + nst - 1) - sk_cta_of_unit(p, u_lo) + 1;
  int last = 0;
  if (lane == 0) last = sk_ticket(p.sk_count + t * 8 + w, static_cast<uint32_t>(nparts)) ? 1 : 0;
  last = __shfl_sync(0xFFFFFFFFu, last, 0);
  if (last) __threadfence();
  return last != 0;
}
// Sum the partials of this warp's region and write them to Y (row m0 + col,
// feature n).  Four groups of 16 columns (16 float4 per thread) per pass: each
// contributor's 16 loads are issued together, so a pass pays one L2 round trip
// per contributor -- the fix-up of a 256-column tile cut in two takes four round
// trips, not sixteen.  The sum runs in CTA order for every value, as before.
template <int CPW>
__device__ __forceinline__ void sk_finish(const TcArgs& p, int64_t t, int nst, int w, int lane, int h, int64_t m0,
                                          int ntok, int64_t n, bool n_ok) {
  constexpr int GB = 4;  // 16-column groups per pass
  static_assert((2 * CPW) % GB == 0, "whole passes");
  const int64_t u_lo = t * nst;
  const int64_t c_lo = sk_cta_of_unit(p, u_lo), c_hi = sk_cta_of_unit(p, u_lo + nst - 1);
#pragma unroll 1
  for (int g0 = 0; g0 < 2 * CPW; g0 += GB) {
    float4 a[GB][4];
#pragma unroll
    for (int gg = 0; gg < GB; ++gg)
#pragma unroll
      for (int k = 0; k < 4; ++k) a[gg][k] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
    for (int64_t c = c_lo; c <= c_hi; ++c) {
      const float4* src = sk_slot(p, c, sk_begin(p, c) >= u_lo, w, lane) + g0 * 4 * 32;
      float4 v[GB][4];
#pragma unroll
      for (int gg = 0; gg < GB; ++gg)
#pragma unroll
        for (int k = 0; k < 4; ++k) v[gg][k] = __ldcg(src + (gg * 4 + k) * 32);
#pragma unroll
      for (int gg = 0; gg < GB; ++gg)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          a[gg][k].x += v[gg][k].x;
          a[gg][k].y += v[gg][k].y;
          a[gg][k].z += v[gg][k].z;
          a[gg][k].w += v[gg][k].w;
        }
    }
    if (n_ok) {
#pragma unroll
      for (int gg = 0; gg < GB; ++gg) {
        const int g = g0 + gg;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int col = (h + 2 * (g >> 1)) * 32 + 16 * (g & 1) + 4 * k;  // float4 q = 4 g + k
          float* yc = p.y + (m0 + col) * p.ldy + n;
          if (col + 0 < ntok) yc[0] = a[gg][k].x;
          if (col + 1 < ntok) yc[p.ldy] = a[gg][k].y;
          if (col + 2 < ntok) yc[2 * p.ldy] = a[gg][k].z;
          if (col + 3 < ntok) yc[3 * p.ldy] = a[gg][k].w;
        }
      }
    }
  }
}

// ------------------------------------------------------------------ roles
template <class SM>
__device__ void producer(const TcArgs& p, SM& S, const CUtensorMap* wmap, const CUtensorMap* amap) {
  const int64_t B = p.K / 32;
  const int nst = static_cast<int>((B + KB - 1) / KB);
  const uint32_t bytes = static_cast<uint32_t>(SM::WROW * TW + SM::ARAW_ROW * p.tt);  // full boxes, zero fill included
  uint32_t gstage = 0;
  SegIter si = seg_iter(p);
  Seg sg;
  while (!S.abort && seg_next(p, nst, si, sg)) {
    const Tile T = decode_tile(p, sg.t);
    for (int s = sg.s0; s < sg.s1; ++s) {
      const int slot = gstage % RAW;
      if (!mbar_wait(&S.empty_raw[slot], ((gstage / RAW) & 1) ^ 1, S)) break;
      mbar_expect_tx(&S.full_raw[slot], bytes);
      if constexpr (SM::WX) {  // 4 blocks = 8 chunks of 16 bytes x 16 groups of 8 rows
        tma_4d(S.wraw[slot], wmap, 0, 0, static_cast<int32_t>(s * KB * 2), static_cast<int32_t>(T.wrow0 / 8),
               &S.full_raw[slot]);
      } else {
        tma_2d(S.wraw[slot], wmap, static_cast<int32_t>(s * KB * 16), static_cast<int32_t>(T.wrow0), &S.full_raw[slot]);
      }
      if constexpr (SM::AX) {  // the activations' operand bytes, same 4D layout as the weights
        tma_4d(S.araw[slot], amap, 0, 0, static_cast<int32_t>(s * KB * 2), static_cast<int32_t>(T.m0 / 8),
               &S.full_raw[slot]);
      } else {
        tma_2d(S.araw[slot], amap, static_cast<int32_t>(s * SM::ARAW_ROW), static_cast<int32_t>(T.m0),
               &S.full_raw[slot]);
      }
      ++gstage;
    }
  }
  // Drain: the last RAW stages' copies must have landed before the CTA exits
  // (normally the consumers already waited for them and this returns at once).
  const uint32_t first = gstage > RAW ? gstage - RAW : 0;
  for (uint32_t g = first; g < gstage; ++g) {
    const uint64_t t0 = gtime();
    while (!mbar_try(&S.full_raw[g % RAW], (g / RAW) & 1) && gtime() - t0 < kTimeoutNs) {
    }
  }
}

template <class SM>
__device__ void mma_issuer(const TcArgs& p, SM& S, uint32_t tmem) {
  const int64_t B = p.K / 32;
  const int nst = static_cast<int>((B + KB - 1) / KB);
  uint32_t gblk = 0;
  uint32_t gst = 0;  // raw stages of the finished segments (the producer's stage order)
  SegIter si = seg_iter(p);
  Seg sg;
  while (seg_next(p, nst, si, sg)) {
    const Tile T = decode_tile(p, sg.t);
    const uint32_t idesc = SM::ABITS == 16 ? bf16_idesc(T.nmma) : f8_idesc(T.nmma);
    const int64_t b_end = static_cast<int64_t>(sg.s1) * KB < B ? static_cast<int64_t>(sg.s1) * KB : B;
    for (int64_t b = static_cast<int64_t>(sg.s0) * KB; b < b_end; ++b, ++gblk) {
      const int f = gblk % SM::F8;
      const int tb = static_cast<int>(gblk % SM::NBUF);
      if constexpr (SM::AX) {  // both operands come straight from the raw stage: wait for its copies
        const int s = static_cast<int>(b / KB);
        const uint32_t g = gst + static_cast<uint32_t>(s - sg.s0);
        if (b == static_cast<int64_t>(s) * KB && !mbar_spin(&S.full_raw[g % RAW], (g / RAW) & 1, S)) goto done;
      } else {
        if (!mbar_spin(&S.f8_full[f], (gblk / SM::F8) & 1, S)) goto done;
      }
      if (!mbar_spin(&S.tm_empty[tb], ((gblk / SM::NBUF) & 1) ^ 1, S)) goto done;
      tc_fence_after();
      const uint32_t dt = tmem + static_cast<uint32_t>(tb * SM::TT);
      if constexpr (SM::AX) {
        const int s = static_cast<int>(b / KB), kb = static_cast<int>(b - static_cast<int64_t>(s) * KB);
        const uint32_t slot = (gst + static_cast<uint32_t>(s - sg.s0)) % RAW;
        mma_f8(dt, kmajor_desc_sbo(S.wraw[slot] + kb * 256, KB * 2 * 128),
               kmajor_desc_sbo(S.araw[slot] + kb * 256, KB * 2 * 128), idesc);
      } else if constexpr (SM::ABITS == 4 && SM::WX) {
        // A straight from the raw stage: block kb's two 16-byte chunks of every
        // row are core matrices 128 bytes apart, 8-row groups 8 chunks apart
        const int s = static_cast<int>(b / KB), kb = static_cast<int>(b - static_cast<int64_t>(s) * KB);
        const uint32_t slot = (gst + static_cast<uint32_t>(s - sg.s0)) % RAW;
        mma_f8(dt, kmajor_desc_sbo(S.wraw[slot] + kb * 256, KB * 2 * 128), kmajor_desc(S.af8[f]), idesc);
      } else if constexpr (SM::ABITS == 4) {
        mma_f8(dt, kmajor_desc(S.wf8[f]), kmajor_desc(S.af8[f]), idesc);
      } else {  // two K = 16 halves of the block (core-matrix pairs 256 bytes apart)
        const uint64_t ad = kmajor_desc_sbo(S.wf8[f], 512), bd = kmajor_desc_sbo(S.af8[f], 512);
        mma_f16(dt, ad, bd, idesc, 0u);
        mma_f16(dt, ad + (256 >> 4), bd + (256 >> 4), idesc, 1u);
      }
      mma_commit(&S.tm_full[tb]);
      if constexpr (!SM::AX) mma_commit(&S.f8_empty[f]);
      if constexpr (SM::WX) {  // the stage's weights are read once its last block's MMA completes
        const int64_t s = b / KB;
        const int64_t last = ((s + 1) * KB < B ? (s + 1) * KB : B) - 1;
        if (b == last) mma_commit(&S.empty_raw[(gst + static_cast<uint32_t>(s - sg.s0)) % RAW]);
      }
    }
    gst += static_cast<uint32_t>(sg.s1 - sg.s0);
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

// f16x2 of two int4 codes (the low nibbles of the bytes `sel` picks from w, as
// q - 8) and of two int8 codes (bytes of x = codes ^ 0x80, as the signed value):
// prmt places each byte under the f16 exponent byte 0x64 (the value 1024 + byte),
// then one exact f16x2 subtraction removes the offset.
__device__ __forceinline__ uint32_t f16x2_sub(uint32_t h, uint32_t c) {
  __half2 a, b;
  memcpy(&a, &h, 4);
  memcpy(&b, &c, 4);
  const __half2 r = __hsub2(a, b);
  uint32_t out;
  memcpy(&out, &r, 4);
  return out;
}
__device__ __forceinline__ uint32_t q4_pair_f16(uint32_t w, uint32_t sel) {
  return f16x2_sub(prmt(w, 0x64646464u, sel) & 0xFF0FFF0Fu, 0x64086408u);  // - 1032
}
__device__ __forceinline__ uint32_t s8_pair_f16(uint32_t x, uint32_t sel) {
  return f16x2_sub(prmt(x, 0x64646464u, sel), 0x64806480u);  // - 1152
}
// bf16x2 of two int4 codes as q - 8: the nibble under the bf16 exponent byte
// 0x43 is 128 + q (7 stored mantissa bits hold 0..15), minus 136 (0x4308),
// exactly.
__device__ __forceinline__ uint32_t q4_pair_bf16(uint32_t w, uint32_t sel) {
  __nv_bfloat162 a, b;
  const uint32_t h = prmt(w, 0x43434343u, sel) & 0xFF0FFF0Fu, c = 0x43084308u;
  memcpy(&a, &h, 4);
  memcpy(&b, &c, 4);
  const __nv_bfloat162 r = __hsub2(a, b);
  uint32_t out;
  memcpy(&out, &r, 4);
  return out;
}

// Stage s's four scales of one row: a vector load when the row's groups are
// aligned, else four clamped scalar loads (validity is applied when stored).
__device__ __forceinline__ uint4 load_scales4(const float* row, int s, int B, bool vec) {
  if (vec) return __ldg(reinterpret_cast<const uint4*>(row + s * KB));
  uint32_t v[KB];
#pragma unroll
  for (int k = 0; k < KB; ++k) v[k] = __float_as_uint(__ldg(row + min(s * KB + k, B - 1)));
  return make_uint4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ uint2 load_halves4(const uint16_t* row, int s, int B, bool vec) {
  if (vec) return __ldg(reinterpret_cast<const uint2*>(row + s * KB));
  uint32_t v[KB];
#pragma unroll
  for (int k = 0; k < KB; ++k) v[k] = __ldg(row + min(s * KB + k, B - 1));
  return make_uint2(v[0] | (v[1] << 16), v[2] | (v[3] << 16));
}

// Two warps convert one stage (4 blocks) at a time.  Thread ct always takes
// block k = ct % 4 of rows r0 + 16 i (r0 = ct / 4): 8 lanes read one row's 64
// contiguous raw bytes, and the lanes of one block write 8 consecutive 16-byte
// core-matrix rows of its fp8 buffer (the buffers are padded so that the four
// blocks' stores land in distinct banks).  Source and destination advance by
// constant strides (16 rows = 1024 raw bytes = 512 fp8 bytes per half).
template <class SM>
__device__ void converters(const TcArgs& p, SM& S) {
  constexpr int F8 = SM::F8;
  constexpr int RS = 8 * SM::CONV;  // rows per pass (a multiple of 8)
  // converter threads: warps 2-3, then warps 12-15 where present
  const int ct = threadIdx.x < 128 ? threadIdx.x - 64 : 64 + threadIdx.x - 384;
  const int lane = threadIdx.x & 31;
  const int k = ct & 3;
  const int r0 = ct >> 2;
  constexpr int AROW = SM::ARAW_ROW;        // raw activation bytes per row and stage
  constexpr int SBO = 256 * SM::OPB;        // operand bytes per 8-row group of a block
  const uint32_t src_off = static_cast<uint32_t>(r0 * (KB * 16) + k * 16);
  const uint32_t asrc_off = static_cast<uint32_t>(r0 * AROW + k * (AROW / KB));
  const uint32_t dst_off = static_cast<uint32_t>((r0 >> 3) * SBO + (r0 & 7) * 16);
  const int64_t B = p.K / 32;
  const int nst = static_cast<int>((B + KB - 1) / KB);
  constexpr int CT = 32 * SM::CONV;             // converter threads
  constexpr int AR = (SM::TT + CT - 1) / CT;    // activation scale rows per thread
  constexpr int WR = (TW + CT - 1) / CT;        // weight scale rows per thread
  // rows whose 4-block groups are aligned take one vector load per array
  const bool vec = (B % KB) == 0 && (reinterpret_cast<uintptr_t>(p.a_scales) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(p.w_scales) & 7) == 0 &&
                   (reinterpret_cast<uintptr_t>(p.w_sums) & 7) == 0;
  uint32_t gstage = 0, gblk = 0;
  SegIter si = seg_iter(p);
  Seg sg;
  while (seg_next(p, nst, si, sg)) {
    const Tile T = decode_tile(p, sg.t);
    const int a_iters = (T.nmma - r0 + RS - 1) / RS;
    for (int s = sg.s0; s < sg.s1; ++s, ++gstage) {
      const int nbk = static_cast<int>(B - s * KB < KB ? B - s * KB : KB);
      const int slot = gstage % RAW;
      // this stage's scales: loaded now, stored into slot gstage % NSC once the
      // stage's codes are converted (the loads' latency hides behind that)
      uint4 sa[AR];
      uint2 swd[WR], sws[WR];
      auto load_stage_scales = [&]() {
      if constexpr (SM::ABITS != 16) {  // the rotate-only route has no activation scales
#pragma unroll
      for (int i = 0; i < AR; ++i) {
        const int m = ct + CT * i;
        const int64_t row = T.m0 + (m < T.ntok ? m : 0);
        sa[i] = load_scales4(p.a_scales + row * B, s, static_cast<int>(B), vec);
      }
      }
#pragma unroll
      for (int i = 0; i < WR; ++i) {
        const int n = ct + CT * i;
        const int64_t row = T.wrow0 + (n < T.rows_w ? n : 0);
        swd[i] = load_halves4(p.w_scales + row * B, s, static_cast<int>(B), vec);
        sws[i] = load_halves4(reinterpret_cast<const uint16_t*>(p.w_sums) + row * B, s, static_cast<int>(B), vec);
      }
      };
      // with nothing to convert the loads wait until the stage has landed (several
      // stages of slack), so that they are not held across the wait
      if constexpr (SM::CONV_SCALES && !SM::AX) load_stage_scales();
      if (!mbar_wait(&S.full_raw[slot], (gstage / RAW) & 1, S)) return;
      if constexpr (SM::AX) load_stage_scales();
      if constexpr (!SM::AX) {  // (expanded operands: nothing to convert, scales only)
      for (int kk = 0; kk < nbk; ++kk) {
        const uint32_t g = gblk + kk;
        if (!mbar_wait(&S.f8_empty[g % F8], ((g / F8) & 1) ^ 1, S)) return;
      }
      if (k < nbk) {
        const int f = (gblk + k) % F8;
        // weights: 128 rows, signed q - 8
        const uint8_t* ws = S.wraw[slot] + src_off;
        uint8_t* wd = S.wf8[f] + dst_off;
        if constexpr (SM::ABITS == 16) {
          // bf16 operands, same layout as the f16 ones: weights q - 8 ...
#pragma unroll 4
          for (int i = 0; i < (TW - r0 + RS - 1) / RS; ++i) {
            const uint4 raw = *reinterpret_cast<const uint4*>(ws + i * RS * 64);
            const uint32_t hx = raw.x >> 4, hy = raw.y >> 4, hz = raw.z >> 4, hw = raw.w >> 4;
            uint8_t* d = wd + i * RS * 64;
            *reinterpret_cast<uint4*>(d) = make_uint4(q4_pair_bf16(raw.x, 0x4140u), q4_pair_bf16(raw.x, 0x4342u),
                                                      q4_pair_bf16(raw.y, 0x4140u), q4_pair_bf16(raw.y, 0x4342u));
            *reinterpret_cast<uint4*>(d + 128) = make_uint4(q4_pair_bf16(raw.z, 0x4140u), q4_pair_bf16(raw.z, 0x4342u),
                                                            q4_pair_bf16(raw.w, 0x4140u), q4_pair_bf16(raw.w, 0x4342u));
            *reinterpret_cast<uint4*>(d + 256) = make_uint4(q4_pair_bf16(hx, 0x4140u), q4_pair_bf16(hx, 0x4342u),
                                                            q4_pair_bf16(hy, 0x4140u), q4_pair_bf16(hy, 0x4342u));
            *reinterpret_cast<uint4*>(d + 384) = make_uint4(q4_pair_bf16(hz, 0x4140u), q4_pair_bf16(hz, 0x4342u),
                                                            q4_pair_bf16(hw, 0x4140u), q4_pair_bf16(hw, 0x4342u));
          }
          // ... and the activations' bf16 values as they are: the block's 64 raw
          // bytes of a row are its four 8-element chunks
          const uint8_t* as = S.araw[slot] + asrc_off;
          uint8_t* ad = S.af8[f] + dst_off;
#pragma unroll 2
          for (int i = 0; i < a_iters; ++i) {
            const uint4* src = reinterpret_cast<const uint4*>(as + i * RS * AROW);
            uint8_t* d = ad + i * RS * 64;
#pragma unroll
            for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(d + 128 * c) = src[c];
          }
        } else if constexpr (SM::ABITS == 8) {
          // f16 operands: chunk c (elements 8c..8c+7) at c * 128; a code q becomes
          // the f16 1024 + q (exponent byte 0x64 above the nibble), minus 1032
#pragma unroll 4
          for (int i = 0; i < (TW - r0 + RS - 1) / RS; ++i) {
            const uint4 raw = *reinterpret_cast<const uint4*>(ws + i * RS * 64);
            const uint32_t hx = raw.x >> 4, hy = raw.y >> 4, hz = raw.z >> 4, hw = raw.w >> 4;
            uint8_t* d = wd + i * RS * 64;
            *reinterpret_cast<uint4*>(d) = make_uint4(q4_pair_f16(raw.x, 0x4140u), q4_pair_f16(raw.x, 0x4342u),
                                                      q4_pair_f16(raw.y, 0x4140u), q4_pair_f16(raw.y, 0x4342u));
            *reinterpret_cast<uint4*>(d + 128) = make_uint4(q4_pair_f16(raw.z, 0x4140u), q4_pair_f16(raw.z, 0x4342u),
                                                            q4_pair_f16(raw.w, 0x4140u), q4_pair_f16(raw.w, 0x4342u));
            *reinterpret_cast<uint4*>(d + 256) = make_uint4(q4_pair_f16(hx, 0x4140u), q4_pair_f16(hx, 0x4342u),
                                                            q4_pair_f16(hy, 0x4140u), q4_pair_f16(hy, 0x4342u));
            *reinterpret_cast<uint4*>(d + 384) = make_uint4(q4_pair_f16(hz, 0x4140u), q4_pair_f16(hz, 0x4342u),
                                                            q4_pair_f16(hw, 0x4140u), q4_pair_f16(hw, 0x4342u));
          }
          // activations: int8 codes s become 1024 + (s + 128), minus 1152
          const uint8_t* as = S.araw[slot] + asrc_off;
          uint8_t* ad = S.af8[f] + dst_off;
#pragma unroll 2
          for (int i = 0; i < a_iters; ++i) {
            const uint4 r0v = *reinterpret_cast<const uint4*>(as + i * RS * AROW);
            const uint4 r1v = *reinterpret_cast<const uint4*>(as + i * RS * AROW + 16);
            const uint32_t v[8] = {r0v.x, r0v.y, r0v.z, r0v.w, r1v.x, r1v.y, r1v.z, r1v.w};
            uint8_t* d = ad + i * RS * 64;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint32_t xa = v[2 * c] ^ 0x80808080u, xb = v[2 * c + 1] ^ 0x80808080u;
              *reinterpret_cast<uint4*>(d + 128 * c) = make_uint4(s8_pair_f16(xa, 0x4140u), s8_pair_f16(xa, 0x4342u),
                                                                  s8_pair_f16(xb, 0x4140u), s8_pair_f16(xb, 0x4342u));
            }
          }
        } else {
        if constexpr (!SM::WX)  // (pre-expanded weights need no conversion)
#pragma unroll 4
        for (int i = 0; i < (TW - r0 + RS - 1) / RS; ++i) {
          const uint4 raw = *reinterpret_cast<const uint4*>(ws + i * RS * 64);
          uint32_t l0, h0, l1, h1, l2, h2, l3, h3;
          q4_0_word_to_e4m3(raw.x, l0, h0);
          q4_0_word_to_e4m3(raw.y, l1, h1);
          q4_0_word_to_e4m3(raw.z, l2, h2);
          q4_0_word_to_e4m3(raw.w, l3, h3);
          *reinterpret_cast<uint4*>(wd + i * RS * 32) = make_uint4(l0, l1, l2, l3);
          *reinterpret_cast<uint4*>(wd + i * RS * 32 + 128) = make_uint4(h0, h1, h2, h3);
        }
        // activations: nmma rows; the offset codes u = a + 8 are the e4m3 bytes
        const uint8_t* as = S.araw[slot] + asrc_off;
        uint8_t* ad = S.af8[f] + dst_off;
#pragma unroll 4
        for (int i = 0; i < a_iters; ++i) {
          const uint4 raw = *reinterpret_cast<const uint4*>(as + i * RS * 64);
          const uint32_t x0 = raw.x ^ 0x88888888u, x1 = raw.y ^ 0x88888888u;
          const uint32_t x2 = raw.z ^ 0x88888888u, x3 = raw.w ^ 0x88888888u;
          *reinterpret_cast<uint4*>(ad + i * RS * 32) =
              make_uint4(x0 & 0x0F0F0F0Fu, x1 & 0x0F0F0F0Fu, x2 & 0x0F0F0F0Fu, x3 & 0x0F0F0F0Fu);
          *reinterpret_cast<uint4*>(ad + i * RS * 32 + 128) = make_uint4(
              (x0 >> 4) & 0x0F0F0F0Fu, (x1 >> 4) & 0x0F0F0F0Fu, (x2 >> 4) & 0x0F0F0F0Fu, (x3 >> 4) & 0x0F0F0F0Fu);
        }
        }
      }
      }
      if constexpr (SM::CONV_SCALES) {
        const int sc = static_cast<int>(gstage % SM::NSC);
#pragma unroll
        for (int i = 0; i < AR; ++i) {
          const int m = ct + CT * i;
          if (m < SM::TT) {
            const bool ok = m < T.ntok;
            uint32_t v[KB] = {0u, 0u, 0u, 0u};
            if constexpr (SM::ABITS != 16) {
              v[0] = sa[i].x; v[1] = sa[i].y; v[2] = sa[i].z; v[3] = sa[i].w;
            }
#pragma unroll
            for (int kk = 0; kk < KB; ++kk)
              S.sda[sc][kk][m] = (ok && kk < nbk) ? (SM::ABITS == 16 ? 1.0f : __uint_as_float(v[kk])) : 0.f;
          }
        }
#pragma unroll
        for (int i = 0; i < WR; ++i) {
          const int n = ct + CT * i;
          if (n < TW) {
            const bool ok = n < T.rows_w;
#pragma unroll
            for (int kk = 0; kk < KB; ++kk) {
              const uint32_t wd2 = kk < 2 ? swd[i].x : swd[i].y, ws2 = kk < 2 ? sws[i].x : sws[i].y;
              const unsigned short dh = static_cast<unsigned short>(wd2 >> (16 * (kk & 1)));
              const short sw = static_cast<short>(ws2 >> (16 * (kk & 1)));
              const bool v = ok && kk < nbk;
              if constexpr (SM::ABITS == 4) {
                const float dw = v ? __half2float(__ushort_as_half(dh)) * fp8_unscale() : 0.f;
                S.sdw[sc][kk][n] = dw;
                // -d_w * 8 S_w, exact: (d_w 2^18) * (S_w 2^-15), at most 20 significant bits
                S.scorr[sc][kk][n] = v ? -dw * (static_cast<float>(sw) * 3.0517578125e-05f) : 0.f;
              } else {  // f16 operands: D is P itself, no offset to remove
                S.sdw[sc][kk][n] = v ? __half2float(__ushort_as_half(dh)) : 0.f;
                S.scorr[sc][kk][n] = 0.f;
              }
            }
          }
        }
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        if constexpr (!SM::AX) {
          for (int kk = 0; kk < nbk; ++kk) mbar_arrive(&S.f8_full[(gblk + kk) % F8]);
          mbar_arrive(&S.empty_raw[slot]);
        }
        if constexpr (SM::CONV_SCALES) mbar_arrive(&S.sc_ready[gstage % SM::NSC]);
      }
      gblk += nbk;
    }
  }
}

template <bool PARTIALS, class SM>
__device__ void workers(const TcArgs& p, SM& S, uint32_t tmem) {
  constexpr int TT = SM::TT;
  constexpr int CPW = TT / 64;  // 32-column chunks per worker warp: h + 2i, i < CPW
  const int wt = threadIdx.x - 128;  // 0..255
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;  // 4..11
  const int q = warp & 3;             // TMEM lane quarter this warp may access
  const int h = (warp - 4) >> 2;      // column half: chunks h, h+2, h+4, h+6
  const int n_in = 32 * q + lane;     // this thread's weight row within the tile
  const int B = static_cast<int>(p.K / 32);
  const int nst = (B + KB - 1) / KB;
  uint32_t gfold = 0, gsc = 0, gtile = 0;

  SegIter si = seg_iter(p);
  Seg sg;
  for (; seg_next(p, nst, si, sg); ++gtile) {
    // the scale slots are reused across segments: start only when every warp is done
    if (gtile > 0 && !mbar_wait(&S.tile_done, (gtile - 1) & 1, S)) return;
    const Tile T = decode_tile(p, sg.t);
    const int nchunks = T.nmma / 32;
    // scale sources of this thread: activation row wt, weight row wt (wt < 128)
    const bool a_ok = wt < T.ntok;
    const bool w_ok = wt < T.rows_w;
    // element offsets of this thread's scale rows: activation row wt, weight row wt
    const int64_t a_off = (T.m0 + (a_ok ? wt : 0)) * B;
    const int64_t w_off = (T.wrow0 + (w_ok ? wt : 0)) * B;
    // Scales of the next stage, prefetched into registers one stage ahead and kept
    // packed as loaded (no arithmetic on them until they are published, so the
    // warp does not wait for the loads): 4 fp32 d_a, 4 fp16 d_w, 4 int16 S_w.
    uint4 da_r;
    uint2 dw_r, sw_r;
    // Loads are unconditional (clamped to valid addresses); validity is applied
    // when publishing, so nothing consumes a loaded value early.
    // Rows whose KB-block groups are aligned take one vector load per array.
    const bool vec = (B % KB) == 0 && (reinterpret_cast<uintptr_t>(p.a_scales) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(p.w_scales) & 7) == 0 &&
                     (reinterpret_cast<uintptr_t>(p.w_sums) & 7) == 0;
    auto load_scales = [&](int s) {
      if constexpr (SM::CONV_SCALES) return;
      if (vec) {
        da_r = __ldg(reinterpret_cast<const uint4*>(p.a_scales + a_off + s * KB));
        dw_r = __ldg(reinterpret_cast<const uint2*>(p.w_scales + w_off + s * KB));
        sw_r = __ldg(reinterpret_cast<const uint2*>(p.w_sums + w_off + s * KB));
        return;
      }
      uint32_t a[KB], w[KB], u[KB];
#pragma unroll
      for (int k = 0; k < KB; ++k) {
        const int b = min(s * KB + k, B - 1);
        a[k] = __float_as_uint(__ldg(p.a_scales + a_off + b));
        w[k] = __ldg(p.w_scales + w_off + b);
        u[k] = static_cast<uint16_t>(__ldg(p.w_sums + w_off + b));
      }
      da_r = make_uint4(a[0], a[1], a[2], a[3]);
      dw_r = make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
      sw_r = make_uint2(u[0] | (u[1] << 16), u[2] | (u[3] << 16));
    };
    // Store the registers' scales into a slot and arrive; waiting is separate.
    auto publish_scales = [&](int slot, int s) {
      if constexpr (SM::CONV_SCALES) return;
      const uint32_t da[KB] = {da_r.x, da_r.y, da_r.z, da_r.w};
      const uint32_t dwp[2] = {dw_r.x, dw_r.y}, swp[2] = {sw_r.x, sw_r.y};
#pragma unroll
      for (int k = 0; k < KB; ++k) {
        const bool bok = s * KB + k < B;
        if (wt < TT) S.sda[slot][k][wt] = (a_ok && bok) ? __uint_as_float(da[k]) : 0.f;
        if (wt < TW) {
          const unsigned short dh = static_cast<unsigned short>(dwp[k >> 1] >> (16 * (k & 1)));
          const short sw = static_cast<short>(swp[k >> 1] >> (16 * (k & 1)));
          const float dw = (w_ok && bok) ? __half2float(__ushort_as_half(dh)) * fp8_unscale() : 0.f;
          S.sdw[slot][k][wt] = dw;
          // -d_w * 8 S_w, exact: (d_w 2^18) * (S_w 2^-15), at most 20 significant bits
          S.scorr[slot][k][wt] = (w_ok && bok) ? -dw * (static_cast<float>(sw) * 3.0517578125e-05f) : 0.f;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.sc_ready[slot]);
    };
    float2 acc[CPW][16];  // column pairs (2j, 2j + 1) of chunk h + 2i
#pragma unroll
    for (int i = 0; i < CPW; ++i)
#pragma unroll
      for (int j = 0; j < 16; ++j) acc[i][j] = make_float2(0.f, 0.f);

    // Stage s's scales live in slot (gsc0 + s - s0) % NSC (see Smem::NSC for
    // who writes them); a stage's slot is waited for at its first block.  When
    // the workers publish, the registers hold stage s + 1's scales during stage s.
    const uint32_t gsc0 = gsc;
    if constexpr (!SM::CONV_SCALES) {
      load_scales(sg.s0);
      publish_scales(static_cast<int>(gsc0 % SM::NSC), sg.s0);
      if (sg.s0 + 1 < sg.s1) load_scales(sg.s0 + 1);
    }

    const int b_end = sg.s1 * KB < B ? sg.s1 * KB : B;
    for (int b = sg.s0 * KB; b < b_end; ++b) {
      const int s = b / KB;
      const int kb = b - s * KB;
      const uint32_t gs = gsc0 + static_cast<uint32_t>(s - sg.s0);
      if (kb == 0 && !mbar_wait(&S.sc_ready[gs % SM::NSC], (gs / SM::NSC) & 1, S)) return;
      // ---- fold block b
      const int tb = static_cast<int>(gfold % SM::NBUF);
      if (!mbar_wait(&S.tm_full[tb], (gfold / SM::NBUF) & 1, S)) return;
      tc_fence_after();
      if (!SM::CONV_SCALES && kb == 2 && s + 1 < sg.s1) {
        publish_scales(static_cast<int>((gs + 1) % SM::NSC), s + 1);
        if (s + 2 < sg.s1) load_scales(s + 2);
      }
      const int slot = static_cast<int>(gs % SM::NSC);
      const float dw = S.sdw[slot][kb][n_in];
      const float corr = S.scorr[slot][kb][n_in];
      const float2 dw2 = make_float2(dw, dw);
      const float2 corr2 = make_float2(corr, corr);
      const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(tb * TT);
      // The buffer goes back to the MMA as soon as this warp's last TMEM load has
      // landed (the fast paths below), not after the folding that follows it.
      bool released = false;
      auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.tm_empty[tb]);
        released = true;
      };
      if (!PARTIALS && TT == 128) {
        // 128-column instance, any tile width: this warp's chunks h and h + 2
        // (those below nchunks) are loaded together, one TMEM round trip per
        // block, then folded.  Columns past ntok inside a chunk are computed and
        // never stored.
        const uint32_t tw = tbase + static_cast<uint32_t>(h * 32);
        const float* dab = &S.sda[slot][kb][h * 32];
        const bool c0 = h < nchunks, c1 = h + 2 < nchunks;
        uint32_t ra[32], rb[32];
        if (c0) tmem_ld32(tw, ra);
        if (c1) tmem_ld32(tw + 64u, rb);
        tmem_wait32x2(ra, rb);
        release();
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (i == 0 ? !c0 : !c1) continue;
          const uint32_t(&cur)[32] = i ? rb : ra;
          const float4* da4 = reinterpret_cast<const float4*>(dab + 64 * i);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 d = da4[j];
            const float2 t0 = __ffma2_rn(
                make_float2(__uint_as_float(cur[4 * j + 0]), __uint_as_float(cur[4 * j + 1])), dw2, corr2);
            const float2 t1 = __ffma2_rn(
                make_float2(__uint_as_float(cur[4 * j + 2]), __uint_as_float(cur[4 * j + 3])), dw2, corr2);
            acc[i][2 * j + 0] = __ffma2_rn(t0, make_float2(d.x, d.y), acc[i][2 * j + 0]);
            acc[i][2 * j + 1] = __ffma2_rn(t1, make_float2(d.z, d.w), acc[i][2 * j + 1]);
          }
        }
      } else if (!PARTIALS && TT == 256 && nchunks == TT / 32) {
        // Full 256-column tile: straight-line fold, TMEM columns and d_a addresses
        // at fixed offsets from this warp's base (chunk h + 2i, piece half).
        const uint32_t tw = tbase + static_cast<uint32_t>(h * 32);
        const float* dab = &S.sda[slot][kb][h * 32];
        uint32_t ra[16], rb[16];
        tmem_ld16(tw, ra);
        tmem_wait(ra);
#pragma unroll
        for (int k = 0; k < 2 * CPW; ++k) {
          uint32_t(&cur)[16] = (k & 1) ? rb : ra;
          uint32_t(&nxt)[16] = (k & 1) ? ra : rb;
          if (k < 2 * CPW - 1) tmem_ld16(tw + static_cast<uint32_t>(64 * ((k + 1) >> 1) + 16 * ((k + 1) & 1)), nxt);
          const int i = k >> 1, half = k & 1;
          const float4* da4 = reinterpret_cast<const float4*>(dab + 64 * i + 16 * half);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float4 d = da4[j];
            const int o = 8 * half + 2 * j;
            const float2 t0 = __ffma2_rn(
                make_float2(__uint_as_float(cur[4 * j + 0]), __uint_as_float(cur[4 * j + 1])), dw2, corr2);
            const float2 t1 = __ffma2_rn(
                make_float2(__uint_as_float(cur[4 * j + 2]), __uint_as_float(cur[4 * j + 3])), dw2, corr2);
            acc[i][o + 0] = __ffma2_rn(t0, make_float2(d.x, d.y), acc[i][o + 0]);
            acc[i][o + 1] = __ffma2_rn(t1, make_float2(d.z, d.w), acc[i][o + 1]);
          }
          if (k < 2 * CPW - 1) {
            tmem_wait(nxt);
            if (k == 2 * CPW - 2) release();  // every piece of this block is in registers
          }
        }
      } else {
        // This warp's 16-column pieces: k -> chunk h + 2 (k / 2), half k % 2.
        // The load of piece k + 1 is in flight while piece k is folded.
        const int npieces = 2 * ((nchunks - h + 1) / 2);
        uint32_t ra[16], rb[16];
        tmem_ld16(tbase + static_cast<uint32_t>(h * 32), ra);
        tmem_wait(ra);
  #pragma unroll
        for (int k = 0; k < 2 * CPW; ++k) {
          if (k < npieces) {
            uint32_t(&cur)[16] = (k & 1) ? rb : ra;
            uint32_t(&nxt)[16] = (k & 1) ? ra : rb;
            const int kn = k + 1;
            if (kn < npieces) tmem_ld16(tbase + static_cast<uint32_t>((h + 2 * (kn >> 1)) * 32 + 16 * (kn & 1)), nxt);
            const int i = k >> 1, half = k & 1;
            const int c0 = (h + 2 * i) * 32 + 16 * half;  // first column of the piece
            if constexpr (PARTIALS) {
              const int64_t n = T.n0 + n_in;
  #pragma unroll 1
              for (int j = 0; j < 16; ++j) {
                const int col = c0 + j;
                if (col < T.ntok && n_in < T.rows_w) {
                  const int64_t m = T.m0 + col;
                  if constexpr (SM::ABITS == 4) {
                    // D = P + 8 S_w, an exact integer times 2^-18
                    const int sw = p.w_sums[(T.wrow0 + n_in) * B + b];
                    p.P[(m * p.N + n) * B + b] =
                        static_cast<int32_t>(__uint_as_float(cur[j]) * fp8_unscale()) - 8 * sw;
                  } else {  // D = P, an exact integer
                    p.P[(m * p.N + n) * B + b] = static_cast<int32_t>(__uint_as_float(cur[j]));
                  }
                }
              }
            } else {
              const float4* da4 = reinterpret_cast<const float4*>(&S.sda[slot][kb][c0]);
  #pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float4 d = da4[j];  // d_a of columns c0 + 4j .. c0 + 4j + 3
                const int o = 8 * half + 2 * j;
                // f32x2 fused multiply-adds: each lane rounds exactly like fmaf
                const float2 t0 = __ffma2_rn(
                    make_float2(__uint_as_float(cur[4 * j + 0]), __uint_as_float(cur[4 * j + 1])), dw2, corr2);
                const float2 t1 = __ffma2_rn(
                    make_float2(__uint_as_float(cur[4 * j + 2]), __uint_as_float(cur[4 * j + 3])), dw2, corr2);
                acc[i][o + 0] = __ffma2_rn(t0, make_float2(d.x, d.y), acc[i][o + 0]);
                acc[i][o + 1] = __ffma2_rn(t1, make_float2(d.z, d.w), acc[i][o + 1]);
              }
            }
            if (kn < npieces) tmem_wait(nxt);
          }
        }
      }
      if (!released) release();
      ++gfold;
    }
    gsc = gsc0 + static_cast<uint32_t>(sg.s1 - sg.s0);

    if constexpr (!PARTIALS) {
      // a tile cut by the stream-K ranges is written by its last contributor
      const bool split = p.sk_units && (sg.s0 > 0 || sg.s1 < nst);
      if (split) {
        float4* mine = sk_slot(p, blockIdx.x, sg.first, warp - 4, lane);
#pragma unroll
        for (int qq = 0; qq < 8 * CPW; ++qq) {
          const int i = qq >> 3, j = 2 * (qq & 7);
          __stcg(mine + qq * 32, make_float4(acc[i][j].x, acc[i][j].y, acc[i][j + 1].x, acc[i][j + 1].y));
        }
        if (sk_arrive(p, sg.t, nst, warp - 4, lane))
          sk_finish<CPW>(p, sg.t, nst, warp - 4, lane, h, T.m0, T.ntok, T.n0 + n_in, n_in < T.rows_w);
      } else if (n_in < T.rows_w) {  // (else: the accumulators are dead during the fix-up)
        const int64_t n = T.n0 + n_in;
#pragma unroll
        for (int i = 0; i < CPW; ++i) {
          const int c = h + 2 * i;
          if (c < nchunks) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float v0 = acc[i][j].x, v1 = acc[i][j].y;
              const int col = c * 32 + 2 * j;
              if (col < T.ntok) {
                p.y[(T.m0 + col) * p.ldy + n] = v0;
              }
              if (col + 1 < T.ntok) {
                p.y[(T.m0 + col + 1) * p.ldy + n] = v1;
              }
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.tile_done);
  }
}

template <bool PARTIALS, int TTM, int AB, bool WEXP, bool AEXP>
__global__ void __launch_bounds__(Smem<TTM, AB, WEXP, AEXP>::THREADS, 1)
    w4a4_gemm_tc_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap amap,
                        const TcArgs p) {
  using SmemT = Smem<TTM, AB, WEXP, AEXP>;
  // Smem is taken straight from the __shared__ array (no integer round trip), so
  // the compiler keeps every access in the shared address space (LDS/STS).  The
  // operands need 16-byte alignment (no swizzle), the TMA boxes 128 bytes.
  extern __shared__ __align__(1024) uint8_t smem_dyn[];
  SmemT& S = *reinterpret_cast<SmemT*>(smem_dyn);
  const int warp = threadIdx.x >> 5;
  if ((static_cast<uint32_t>(__cvta_generic_to_shared(smem_dyn)) & 127u) != 0) {  // never expected
    if (threadIdx.x == 0) atomicOr(&g_w4a4_device_error, 2);
    return;
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < RAW; ++i) {
      mbar_init(&S.full_raw[i], 1);
      // the converters' arrivals (unless nothing is converted), plus the MMA's commit when it reads the stage
      mbar_init(&S.empty_raw[i], (SmemT::AX ? 0 : SmemT::CONV) + (SmemT::WX ? 1 : 0));
    }
    for (int i = 0; i < SmemT::F8; ++i) {
      mbar_init(&S.f8_full[i], SmemT::CONV);
      mbar_init(&S.f8_empty[i], 1);
    }
    for (int i = 0; i < SmemT::NBUF; ++i) {
      mbar_init(&S.tm_full[i], 1);
      mbar_init(&S.tm_empty[i], kWorkerWarps);
    }
    for (int i = 0; i < SmemT::NSC; ++i) mbar_init(&S.sc_ready[i], SmemT::CONV_SCALES ? SmemT::CONV : kWorkerWarps);
    mbar_init(&S.tile_done, kWorkerWarps);
    mbar_init(&S.mma_done, 1);
    S.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&wmap)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&amap)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&S.tmem_base)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp < 4 || warp >= 12) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(SmemT::REGS_LOW));
    if (warp == 0) {
      if ((threadIdx.x & 31) == 0) producer(p, S, &wmap, &amap);
      __syncwarp();
    } else if (warp == 1) {
      if ((threadIdx.x & 31) == 0) mma_issuer(p, S, tmem);
      __syncwarp();
    } else {
      converters(p, S);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(SmemT::REGS_HIGH));
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

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2D map over packed codes [rows][K/2] bytes, box = 64 bytes x box_rows rows.
cudaError_t codes_map(CUtensorMap* m, const uint8_t* codes, int64_t rows, int64_t K, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(KB * 16), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(codes), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 4D map over the expanded weights [rows8][K] bytes that writes a box straight in
// the K-major operand layout: dims {16 bytes, 8 rows of a group, K/16 chunks,
// rows8/8 groups}, strides {K, 16, 8K} bytes; a box of 4 blocks (8 chunks) x
// box_rows rows lands as [group][chunk][row][16 bytes].
cudaError_t expanded_map(CUtensorMap* m, const uint8_t* wexp, int64_t rows, int64_t K, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const int64_t groups = (rows + 7) / 8;
  const cuuint64_t dims[4] = {16, 8, static_cast<cuuint64_t>(K / 16), static_cast<cuuint64_t>(groups)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(K), 16, static_cast<cuuint64_t>(8 * K)};
  const cuuint32_t box[4] = {16, 8, static_cast<cuuint32_t>(KB * 2), static_cast<cuuint32_t>(box_rows / 8)};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<uint8_t*>(wexp), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <bool PARTIALS, int TTM, int AB = 4, bool WEXP = false, bool AEXP = false>
cudaError_t launch_tc(const CUtensorMap& wmap, const CUtensorMap& amap, const TcArgs& a, int64_t max_tiles,
                      cudaStream_t stream) {
  auto kern = w4a4_gemm_tc_kernel<PARTIALS, TTM, AB, WEXP, AEXP>;
  using SM = Smem<TTM, AB, WEXP, AEXP>;
  constexpr size_t kSmemBytes = sizeof(SM);
  static bool configured[64] = {};
  static int regs_ok[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    // setmaxnreg.inc waits until the block's launch registers cover the split:
    // refuse to launch a build whose register count would make it wait forever.
    cudaFuncAttributes fa{};
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    const int low_threads = SM::THREADS - 256;  // warpgroup 0 (and 3)
    regs_ok[dev] = (fa.numRegs * SM::THREADS >= low_threads * SM::REGS_LOW + 256 * SM::REGS_HIGH) ? 1 : -1;
    configured[dev] = true;
  }
  if (regs_ok[dev] < 0) return cudaErrorInvalidConfiguration;
  int64_t grid = max_tiles < num_sms() ? max_tiles : num_sms();
  if (grid < 1) grid = 1;
  kern<<<static_cast<unsigned>(grid), SM::THREADS, kSmemBytes, stream>>>(wmap, amap, a);
  return cudaGetLastError();
}

// Token tile of the dense product (the kernel instance's TTM).
#ifndef W4A4_DENSE_TT
#define W4A4_DENSE_TT 256
#endif
constexpr int kDenseTT = W4A4_DENSE_TT;

int token_tile(int64_t M, int ttm) {
  const int64_t r = (M + 31) & ~int64_t(31);
  return static_cast<int>(r < ttm ? r : ttm);
}

// Stream-K or one tile per CTA pass.  Whole tiles leave SMs idle in the last
// wave (80 tiles of M512 x N5120 on 152 SMs: one wave at 53%); stream-K gives
// every CTA the same number of K stages and pays for it with one partial
// store + reload per cut tile.  It is used where it shortens the longest CTA
// by more than 10% (fixup counted as two stages).
struct SkPlan {
  bool on;
  int64_t units;
  int grid;
  size_t count_bytes;  // the ticket region
  size_t ws_bytes;     // tickets + partials
};
constexpr int kSkFixupStages = 2;
// The tickets sit in a fixed region at the start of the workspace, the same for
// every shape, so that partials written for one shape never land on the tickets
// of another when callers reuse one workspace across shapes.
constexpr int64_t kSkMaxTiles = 32768;
constexpr size_t kSkTicketBytes = static_cast<size_t>(kSkMaxTiles) * 8 * sizeof(uint32_t);  // 1 MiB
constexpr size_t kSkPartBytes = size_t(8) * 1024 * sizeof(float4);  // one CTA segment: 8 warps x 32 x 32 float4

SkPlan plan_stream_k(int64_t M, int64_t N, int64_t K, int ttm = kDenseTT) {
  SkPlan pl{};
  if (M <= 0 || N <= 0 || K <= 0) return pl;
  const int64_t tt = token_tile(M, ttm);
  const int64_t tiles = ((N + TW - 1) / TW) * ((M + tt - 1) / tt);
  const int64_t nst = (K / 32 + KB - 1) / KB;
  const int64_t sms = num_sms();
  const int64_t dp_span = ((tiles + sms - 1) / sms) * nst;
  const int64_t U = tiles * nst;
  const int64_t G = U < sms ? U : sms;
  const int64_t sk_span = (U + G - 1) / G + kSkFixupStages;
  if (G < 2 || tiles > kSkMaxTiles || 10 * sk_span >= 9 * dp_span) return pl;
  pl.on = true;
  pl.units = U;
  pl.grid = static_cast<int>(G);
  pl.count_bytes = kSkTicketBytes;
  pl.ws_bytes = pl.count_bytes + 2 * static_cast<size_t>(G) * kSkPartBytes;
  return pl;
}

}  // namespace

// The exact path's product runs the 128-column instance with int8 activations.
constexpr int kW4A8TT = 128;

size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) { return plan_stream_k(M, N, K).ws_bytes; }
size_t gemm_w4a8_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  return plan_stream_k(M, N, K, kW4A8TT).ws_bytes;
}

cudaError_t encode_2d_map(CUtensorMap* m, CUtensorMapDataType dtype, const void* base, uint64_t inner, uint64_t rows,
                          uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Cached per device for the process's life; cudaDeviceReset invalidates the
// cached address (the header tells callers not to use a reset device again).
int* device_error_word() {
  static std::mutex mu;
  static int* cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_w4a4_device_error) != cudaSuccess) return nullptr;
    cached[dev] = static_cast<int*>(p);
  }
  return cached[dev];
}

cudaError_t launch_gemm_tc(const uint8_t* w_codes, const uint16_t* w_scales, const int16_t* w_sums,
                           const uint8_t* w_expanded, int64_t N, const uint8_t* a_codes, const float* a_scales,
                           int64_t M, int64_t K, float* y, int64_t ldy, int32_t* P, void* ws, size_t ws_bytes,
                           cudaStream_t stream) {
  TcArgs a{};
  a.w_scales = w_scales; a.w_sums = w_sums; a.a_scales = a_scales;
  a.M = M; a.N = N; a.K = K; a.y = y; a.ldy = ldy; a.P = P;
  a.tt = token_tile(M, P ? 256 : kDenseTT);
  const bool wexp = w_expanded != nullptr && !P;
  CUtensorMap wmap, amap;
  cudaError_t e = wexp ? expanded_map(&wmap, w_expanded, N, K, TW) : codes_map(&wmap, w_codes, N, K, TW);
  if (e == cudaSuccess) e = codes_map(&amap, a_codes, M, K, a.tt);
  if (e != cudaSuccess) return e;
  int64_t grid = ((N + TW - 1) / TW) * ((M + a.tt - 1) / a.tt);
  if (P) return launch_tc<true, 256>(wmap, amap, a, grid, stream);
  const SkPlan pl = plan_stream_k(M, N, K);
  if (pl.on && ws && ws_bytes >= pl.ws_bytes) {
    a.sk_units = pl.units;
    a.sk_count = static_cast<uint32_t*>(ws);
    a.sk_part = reinterpret_cast<float4*>(static_cast<uint8_t*>(ws) + pl.count_bytes);
    grid = pl.grid;
  }
  if (wexp) return launch_tc<false, kDenseTT, 4, true>(wmap, amap, a, grid, stream);
  return launch_tc<false, kDenseTT>(wmap, amap, a, grid, stream);
}

cudaError_t launch_gemm_w4a8(const uint8_t* w_codes, const uint16_t* w_scales, const int16_t* w_sums, int64_t N,
                             const int8_t* a_codes, const float* a_scales, int64_t M, int64_t K, float* y, int64_t ldy,
                             int32_t* P, void* ws, size_t ws_bytes, cudaStream_t stream) {
  TcArgs a{};
  a.w_scales = w_scales; a.w_sums = w_sums; a.a_scales = a_scales;
  a.M = M; a.N = N; a.K = K; a.y = y; a.ldy = ldy; a.P = P;
  a.tt = token_tile(M, kW4A8TT);
  CUtensorMap wmap, amap;
  cudaError_t e = codes_map(&wmap, w_codes, N, K, TW);
  // int8 codes [M][K]: box of 4 blocks (128 bytes) x tt rows
  if (e == cudaSuccess)
    e = encode_2d_map(&amap, CU_TENSOR_MAP_DATA_TYPE_UINT8, a_codes, static_cast<uint64_t>(K), static_cast<uint64_t>(M),
                      static_cast<uint64_t>(K), KB * 32, static_cast<uint32_t>(a.tt), CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  int64_t grid = ((N + TW - 1) / TW) * ((M + a.tt - 1) / a.tt);
  if (P) return launch_tc<true, kW4A8TT, 8>(wmap, amap, a, grid, stream);
  const SkPlan pl = plan_stream_k(M, N, K, kW4A8TT);
  if (pl.on && ws && ws_bytes >= pl.ws_bytes) {
    a.sk_units = pl.units;
    a.sk_count = static_cast<uint32_t*>(ws);
    a.sk_part = reinterpret_cast<float4*>(static_cast<uint8_t*>(ws) + pl.count_bytes);
    grid = pl.grid;
  }
  return launch_tc<false, kW4A8TT, 8>(wmap, amap, a, grid, stream);
}

cudaError_t launch_gemm_w4a16(const uint8_t* w_codes, const uint16_t* w_scales, const int16_t* w_sums, int64_t N,
                              const uint16_t* a_bf16, int64_t M, int64_t K, float* y, int64_t ldy, void* ws,
                              size_t ws_bytes, cudaStream_t stream) {
  TcArgs a{};
  a.w_scales = w_scales; a.w_sums = w_sums; a.a_scales = nullptr;
  a.M = M; a.N = N; a.K = K; a.y = y; a.ldy = ldy; a.P = nullptr;
  a.tt = token_tile(M, kW4A8TT);
  CUtensorMap wmap, amap;
  cudaError_t e = codes_map(&wmap, w_codes, N, K, TW);
  // bf16 values [M][K] as bytes: box of 4 blocks (256 bytes) x tt rows
  if (e == cudaSuccess)
    e = encode_2d_map(&amap, CU_TENSOR_MAP_DATA_TYPE_UINT8, a_bf16, static_cast<uint64_t>(2 * K),
                      static_cast<uint64_t>(M), static_cast<uint64_t>(2 * K), KB * 64, static_cast<uint32_t>(a.tt),
                      CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  int64_t grid = ((N + TW - 1) / TW) * ((M + a.tt - 1) / a.tt);
  const SkPlan pl = plan_stream_k(M, N, K, kW4A8TT);
  if (pl.on && ws && ws_bytes >= pl.ws_bytes) {
    a.sk_units = pl.units;
    a.sk_count = static_cast<uint32_t*>(ws);
    a.sk_part = reinterpret_cast<float4*>(static_cast<uint8_t*>(ws) + pl.count_bytes);
    grid = pl.grid;
  }
  return launch_tc<false, kW4A8TT, 16>(wmap, amap, a, grid, stream);
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
