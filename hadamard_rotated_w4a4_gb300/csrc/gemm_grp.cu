// Block-scaled W4A4 GEMM over super-tiles (tcgen05, TMEM, TMA): the dense
// product with the expanded activation operand, and the expert-routed product.
//
// Engine docs "The lean option: ROCmFP4, ROCmI4 and Hadamard Q4_0", section
// "Hadamard-rotated Q4_0: W4A4 prompt processing": int4 weights times int4
// activations on the matrix units, weights read as plain Q4_0 (code q stands for
// q - 8); section "MoE: W4A4 on the experts": the same product on the routed
// expert matmuls (MUL_MAT_ID).
//
//   P[n][m][b] = sum_{j<32} (q_w - 8) a        exact, one fp8 MMA per block
//   Y[m][n]   += d_w[n][b] d_a[m][b] P          fp32 fold on the CUDA cores
//
// Operands (the exact fp8 encoding of the tensor-core GEMM in gemm_tc.cu): the
// weights enter as the e4m3 bytes of (q - 8) 2^-9, converted here from the Q4_0
// codes (or loaded pre-expanded); the activations as their offset codes a + 8,
// bytes that are the e4m3 values (a + 8) 2^-9 -- written beforehand by the
// activation kernel (dense), or expanded here from the routed rows' int4 codes
// (routed).  The MMA gives D = (P + 8 S_w) 2^-18 exactly and the fold computes
//   t = fma(D, d_w 2^18, -d_w 8 S_w) = round(d_w P),   acc = fma(t, d_a, acc).
//
// Super-tile.  A tile is one token segment (up to 256 activation rows, the MMA
// N rounded up to 32 columns, cw) against g <= G consecutive 128-row weight
// tiles of one expert: g MMAs per 32-block share the segment's operand and write
// columns [i cw, (i + 1) cw) of a 256-column TMEM accumulator.  An expert that
// receives ~64 tokens then still fills 256 accumulator columns with 4 weight
// tiles, so the fold works on full blocks.
//
// Fold layout.  Each worker thread reads its accumulators with 16x256b TMEM
// loads: 4 weight rows (its lane quarter's rows j, j + 8, j + 16, j + 24) by 32
// token columns (2 of every 8).  A d_a value in shared memory then serves 4 rows
// instead of 1, and a warp's d_a loads are 32 contiguous bytes (one wavefront).
//
// Warp roles (512 threads; 384 with pre-expanded weights, which need no warps 12-15):
//   warp 0         producer: TMA loads of each stage (4 blocks) into a 3-deep ring;
//   warp 1         TMEM allocator and MMA issuer;
//   warps 2-3      publishers: each stage's scales (d_a, d_w 2^18, -d_w 8 S_w) into a
//                  scale slot;
//   warps 12-15    converters: the operand codes into the fp8 operand, block by block;
//   warps 4-11     workers: the fold of each block, the epilogue.
// Every pipeline wait is bounded; a wait that gives up sets the device error
// word (read by w4a4_check) and the CTA winds down.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "tc_ptx.cuh"
#include "w4a4_kernels.cuh"

namespace w4a4 {

namespace {

constexpr int TW = 128;       // weight rows per sub-tile (MMA M, TMEM lanes)
constexpr int KB = 4;         // 32-blocks per stage
constexpr int RAW = 3;        // raw stages in flight
constexpr int TCOLS = 256;    // accumulator columns of a tile
constexpr int NBUF = 2;       // TMEM accumulator buffers
constexpr uint32_t kTmemCols = 512;
constexpr int kWorkers = 8;   // warps 4-11
constexpr uint64_t kDrainNs = 1000000000ull;  // bound of the wind-down waits (1 s)

// G: weight tiles per tile (1 or 4).  WEXP: the weights come pre-expanded (the
// e4m3 bytes, loaded straight into the operand layout).  AEXP: the activations
// come expanded (offset-code bytes, loaded straight into the operand layout);
// otherwise the converters expand their int4 codes next to the weights.
template <int GT, bool WEXP, bool AEXP>
struct __align__(1024) GSmem {
  static constexpr int G = GT;
  static_assert(G == 1 || !WEXP, "pre-expanded weights with single-weight-tile tiles only");
  static_assert(AEXP || G == 4, "converted activations in the multi-tile instance only");
  static constexpr bool WX = WEXP;
  static constexpr bool AX = AEXP;
  // helper warps (each publishes scales and converts operands): warps 2-3 and
  // 12-15 (the pre-expanded-weight instance converts nothing: warps 2-3 only)
  static constexpr int HELP = WEXP ? 2 : 6;
  static constexpr int PUB = 2;            // publishers: warps 2-3
  static constexpr int CONV = HELP - PUB;  // converters: warps 12-15
  static constexpr int THREADS = WEXP ? 384 : 512;
  static constexpr int REGS_LOW = WEXP ? 56 : 48;     // warpgroups 0 and 3
  static constexpr int REGS_HIGH = WEXP ? 224 : 208;  // warpgroups 1-2 (workers)
  static constexpr int WSUB = WEXP ? 16384 : 8192;      // raw weight bytes per sub-tile and stage
  static constexpr int AROW = AEXP ? 128 : 64;          // raw activation bytes per row and stage
  // a stage holds cw activation rows then g weight sub-tiles, g * cw <= 256, g <= G
  static constexpr int STAGE = G == 1 ? 256 * AROW + WSUB : (AEXP ? 40960 : 36864);
  static constexpr int F8 = WEXP ? 1 : (G == 1 ? 8 : 3);  // converted-operand slots (one block each)
  static constexpr int F8W = G * 4096;                    // weight operand: 128 rows x 32 bytes per sub-tile
  static constexpr int F8B = F8W + (AEXP ? 0 : 8192);     // + the activation operand (<= 256 rows x 32 bytes)
  // scale slots (the workers free a slot after the stage's last block): the converters
  // may publish this many stages ahead of the fold
  static constexpr int NSC = G == 1 ? 4 : 2;
  // [activation rows: cw x AROW bytes in 32-row TMA boxes][weights: g x WSUB]; the
  // expanded operands in the 128-byte swizzle, 1024-byte aligned atoms
  uint8_t raw[RAW][STAGE];
  uint8_t f8[F8][F8B];
  float sda[NSC][KB][TCOLS];    // d_a per column, permuted (see col_slot)
  float sdw[NSC][KB][G][TW];    // d_w 2^18 per weight row, permuted (see row_slot)
  float scorr[NSC][KB][G][TW];  // -d_w 8 S_w
  // output staging of the single-weight-tile instance: per worker warp, 8 tokens x 32
  // features, 16-byte groups XOR-swizzled by token (see store_rows)
  float ystage[G == 1 ? kWorkers : 1][G == 1 ? 256 : 1];
  // (NSC is declared above its use in the arrays)
  uint64_t full_raw[RAW];
  uint64_t empty_raw[RAW];
  uint64_t f8_full[F8];
  uint64_t f8_empty[F8];
  uint64_t tm_full[NBUF];
  uint64_t tm_empty[NBUF];
  uint64_t sc_ready[NSC];
  uint64_t sc_free[NSC];
  uint64_t mma_done;
  uint32_t tmem_base;
  volatile int abort;
};
static_assert(sizeof(GSmem<1, false, true>) <= 227 * 1024, "shared memory per CTA is at most 227 KB");
static_assert(sizeof(GSmem<1, true, true>) <= 227 * 1024, "shared memory per CTA is at most 227 KB");
static_assert(sizeof(GSmem<4, false, true>) <= 227 * 1024, "shared memory per CTA is at most 227 KB");
static_assert(sizeof(GSmem<4, false, false>) <= 227 * 1024, "shared memory per CTA is at most 227 KB");

// d_a of tile column c lives at sda[..][col_slot(c)]: a thread (u = lane % 4)
// reads the 8 values of its columns 32k + 8x + 2u + e (x < 4, e < 2) of chunk k
// as two contiguous float4 at 32k + 8u.
__device__ __forceinline__ int col_slot(int c) {
  return (c & ~31) | (((c >> 1) & 3) << 3) | (((c >> 3) & 3) << 1) | (c & 1);
}
// d_w of weight row r (0..127) lives at row_slot(r): a thread (j = lane / 4) of
// quarter q reads its rows 32q + j + 8s (s < 4) as one float4 at 32q + 4j.
__device__ __forceinline__ int row_slot(int r) { return (r & ~31) | ((r & 7) << 2) | ((r >> 3) & 3); }

struct GArgs {
  const uint16_t* w_scales;  // fp16 [rows][B]
  const int16_t* w_sums;     // int16 [rows][B]: S_w = sum_j (q_w - 8)
  const float* a_scales;     // [activation rows][B]
  float* y;
  int64_t ldy;
  int64_t M;                 // dense: tokens
  int64_t N;                 // output features (per expert)
  int64_t K;
  int NT;                    // weight tiles per expert: ceil(N / 128)
  int dense_g;               // dense: weight tiles per tile
  int64_t dense_nseg;        // dense: token segments of 256
  // routed (null for dense)
  const int4* segs;          // [nseg] {first gathered row, expert, tokens, g}
  const int32_t* seg_tiles;  // [nseg + 1] first tile of each segment
  const int32_t* counts;     // {nseg, ntiles} written by the routing kernel
  const int32_t* perm;       // gathered row -> output row
  // stream-K (dense only): 0 = whole tiles blockIdx.x, blockIdx.x + gridDim.x, ...
  int64_t sk_units;
  uint32_t* sk_count;
  float4* sk_part;
  int sk_dyn;                // routed: stream-K over the routing kernel's tiles (units counted on the device)
  int* err;                  // device error word
  uint64_t wait_ns;          // bound of a pipeline wait
  uint64_t producer_delay_ns;  // test hook: the producer starts this late
};

// ------------------------------------------------------------------ bounded waits
template <class SM>
__device__ __forceinline__ bool give_up(SM& S, const GArgs& p) {
  S.abort = 1;
  atomicOr(p.err, 1);
  return false;
}
template <class SM>
__device__ __forceinline__ bool bwait(uint64_t* b, uint32_t parity, SM& S, const GArgs& p) {
  if (mbar_try(b, parity)) return true;
  const uint64_t t0 = gtime();
  for (;;) {
    if (mbar_try(b, parity)) return true;
    if (S.abort) return false;
    if (gtime() - t0 > p.wait_ns) return give_up(S, p);
  }
}
// Spinning variant for the MMA issuer (non-blocking tests, limits checked every 64 polls).
template <class SM>
__device__ __forceinline__ bool bspin(uint64_t* b, uint32_t parity, SM& S, const GArgs& p) {
  if (mbar_test(b, parity)) return true;
  const uint64_t t0 = gtime();
  for (uint32_t n = 1;; ++n) {
    if (mbar_test(b, parity)) return true;
    if ((n & 63) == 0) {
      if (S.abort) return false;
      if (gtime() - t0 > p.wait_ns) return give_up(S, p);
    }
  }
}
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------------ tiles
struct Tile {
  int64_t a_row0;  // first activation row of the segment
  int64_t wrow0;   // first weight row (stacked experts) of sub-tile 0
  int64_t n0;      // first output feature of sub-tile 0 (within the expert)
  int ntok;        // valid tokens
  int cw;          // columns per sub-tile: ntok rounded up to 32
  int g;           // sub-tiles
};

__device__ __forceinline__ int64_t num_tiles(const GArgs& p) {
  if (p.segs) return p.counts[1];
  return p.dense_nseg * ((p.NT + p.dense_g - 1) / p.dense_g);
}

__device__ __forceinline__ Tile tile_at(const GArgs& p, int64_t t) {
  Tile T;
  if (p.segs) {
    int lo = 0, hi = p.counts[0] - 1;  // last segment whose first tile is <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.seg_tiles[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int4 sg = p.segs[lo];
    const int j = static_cast<int>(t - p.seg_tiles[lo]);
    T.a_row0 = sg.x;
    T.ntok = sg.z;
    T.n0 = static_cast<int64_t>(j) * sg.w * TW;
    T.g = min(sg.w, p.NT - j * sg.w);
    T.wrow0 = static_cast<int64_t>(sg.y) * p.N + T.n0;
  } else {  // weight-group major: consecutive CTAs share a weight group in L2
    const int64_t seg = t % p.dense_nseg, wg = t / p.dense_nseg;
    T.a_row0 = seg * TCOLS;
    const int64_t left = p.M - T.a_row0;
    T.ntok = static_cast<int>(left < TCOLS ? left : TCOLS);
    T.n0 = wg * p.dense_g * TW;
    T.g = static_cast<int>(min(static_cast<int64_t>(p.dense_g), p.NT - wg * p.dense_g));
    T.wrow0 = T.n0;
  }
  T.cw = (T.ntok + 31) & ~31;
  return T;
}

// ------------------------------------------------------------------ schedule
struct Seg {
  int64_t t;
  int s0, s1;
  bool first;
};
// The schedule: U stream-K units (tile x stage) cut into G = min(U, gridDim.x)
// equal ranges, one per CTA below G (the others idle: every range is non-empty,
// so a cut tile's contributors are exactly the CTAs from its first to its last),
// or whole tiles blockIdx.x, blockIdx.x + gridDim.x, ... (U = 0).  Dense: U from
// the host (which launches at most U CTAs); routed with stream-K: ntiles x
// stages, once the routing kernel has written the tile count.
struct Sched {
  int64_t U;
  int64_t ntiles;
  int64_t G;
  bool narrow;  // U x G < 2^32: the plan's products and quotients fit 32-bit arithmetic
};
// a / b for 0 <= a < 2^32 when the plan is narrow (a 64-bit division costs ~10x more)
__device__ __forceinline__ int64_t sk_div(const Sched& sch, int64_t a, int64_t b) {
  return sch.narrow ? static_cast<int64_t>(static_cast<uint32_t>(a) / static_cast<uint32_t>(b)) : a / b;
}
__device__ __forceinline__ Sched make_sched(const GArgs& p, int nst) {
  Sched r;
  r.ntiles = num_tiles(p);
  r.U = p.sk_units;
  if (p.sk_dyn) {  // the dense plan's rule: only where it shortens the longest CTA by more
                   // than 10%, a fix-up counted as two stages (every role decides alike)
    const int64_t G = gridDim.x, U = r.ntiles * nst;
    const int64_t dp_span = ((r.ntiles + G - 1) / G) * nst, sk_span = (U + G - 1) / G + 2;
    r.U = (U >= 2 && 10 * sk_span < 9 * dp_span) ? U : 0;
  }
  r.G = (r.U && r.U < static_cast<int64_t>(gridDim.x)) ? r.U : static_cast<int64_t>(gridDim.x);
  r.narrow = r.U * r.G < (static_cast<int64_t>(1) << 32);
  return r;
}
__device__ __forceinline__ int64_t sk_begin(const Sched& sch, int64_t c) {
  return c >= sch.G ? sch.U : sk_div(sch, c * sch.U, sch.G);
}
__device__ __forceinline__ int64_t seg_start(const Sched& sch) {
  return sch.U ? sk_begin(sch, blockIdx.x) : static_cast<int64_t>(blockIdx.x);
}
__device__ __forceinline__ bool seg_next(const Sched& sch, int nst, int64_t& next, Seg& g) {
  const int64_t U = sch.U, ntiles = sch.ntiles;
  if (U) {
    const int64_t start = sk_begin(sch, blockIdx.x), end = sk_begin(sch, blockIdx.x + 1);
    if (next >= end) return false;
    g.first = next == start;
    g.t = sk_div(sch, next, nst);
    g.s0 = static_cast<int>(next - g.t * nst);
    const int64_t left = end - next;
    g.s1 = (nst - g.s0 <= left) ? nst : g.s0 + static_cast<int>(left);
    next += g.s1 - g.s0;
  } else {
    if (next >= ntiles) return false;
    g.first = next == blockIdx.x;
    g.t = next;
    g.s0 = 0;
    g.s1 = nst;
    next += gridDim.x;
  }
  return true;
}
__device__ __forceinline__ int64_t sk_cta_of_unit(const Sched& sch, int64_t u) {
  const int64_t G = sch.G;
  int64_t c = sk_div(sch, u * G, sch.U);
  if (c >= G) c = G - 1;
  for (int i = 0; i < 4 && c > 0 && sk_begin(sch, c) > u; ++i) --c;
  for (int i = 0; i < 4 && c + 1 < G && sk_begin(sch, c + 1) <= u; ++i) ++c;
  return c;
}
// One arrival on a (tile, warp) ticket: true for the last of `nparts`, which
// also puts the ticket back to zero, so the workspace needs no clearing between
// launches (graph replays included).
__device__ __forceinline__ bool sk_ticket(uint32_t* ctr, uint32_t nparts) {
  const uint32_t before = atomicAdd(ctr, 1u);
  if (before + 1 != nparts) return false;
  atomicExch(ctr, 0u);
  return true;
}
__device__ __forceinline__ float4* sk_slot(const GArgs& p, int64_t cta, bool first, int w, int lane) {
  return p.sk_part + ((2 * cta + (first ? 0 : 1)) * 8 + w) * 1024 + lane;
}

// Loads and adds of stream-K partial tiles (a warp's region: 32 float4 per lane).
__device__ __forceinline__ void sk_load8(const float4* src, int kk, float4 (&v)[2][4]) {
#pragma unroll
  for (int hf = 0; hf < 2; ++hf)
#pragma unroll
    for (int x = 0; x < 4; ++x) v[hf][x] = __ldcg(src + ((kk * 2 + hf) * 4 + x) * 32);
}
__device__ __forceinline__ void sk_add8(float2 (&a)[2][4][2], const float4 (&v)[2][4]) {
#pragma unroll
  for (int hf = 0; hf < 2; ++hf)
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      a[hf][x][0].x += v[hf][x].x;
      a[hf][x][0].y += v[hf][x].y;
      a[hf][x][1].x += v[hf][x].z;
      a[hf][x][1].y += v[hf][x].w;
    }
}
// A relaxed read of a ticket; the fence the reader issues before reading the
// partials it counts completes the acquire.
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Stream-K epilogue of a warp's part of a tile cut between CTAs.  Each
// contributor but the last deposits its part in its partial slot and arrives on
// the tile's ticket; the last sums every part in CTA order, (((p_lo + p_lo+1) +
// ...) + p_hi), taking its own part from its registers where that order allows,
// so the result does not depend on which CTA comes last.  A contributor that
// finds every other part already deposited, and whose own part can be added from
// registers (two parts, or the first of several), is the last without arriving
// and writes no partial.  True if acc now holds the tile's sum (this warp writes
// Y), false if the part was deposited.
__device__ __forceinline__ bool sk_epilogue(const GArgs& p, const Sched& sch, const Seg& sg, int nst, int w, int lane,
                                            float2 (&acc)[4][2][4][2]) {
  const int64_t u_lo = sg.t * nst;
  const int64_t c_lo = sk_cta_of_unit(sch, u_lo), c_hi = sk_cta_of_unit(sch, u_lo + nst - 1);
  const uint32_t nparts = static_cast<uint32_t>(c_hi - c_lo + 1);
  // ticket of this (tile, warp) region: per tile (dense), or per the tile's first
  // CTA (routed: a CTA's range ends inside at most one tile that starts in it)
  uint32_t* ctr = p.sk_count + (p.sk_dyn ? c_lo : sg.t) * 8 + w;
  const int64_t me = blockIdx.x;
  int last = 0;
  // every other part is in and this one can stay in registers: no arrival, reset
  if (lane == 0 && (nparts == 2 || me == c_lo) && ld_relaxed_u32(ctr) + 1 == nparts) {
    atomicExch(ctr, 0u);
    last = 1;
  }
  last = __shfl_sync(0xFFFFFFFFu, last, 0);
  if (!last) {
    float4* mine = sk_slot(p, me, sg.first, w, lane);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int x = 0; x < 4; ++x)
          __stcg(mine + ((kk * 2 + hf) * 4 + x) * 32,
                 make_float4(acc[kk][hf][x][0].x, acc[kk][hf][x][0].y, acc[kk][hf][x][1].x, acc[kk][hf][x][1].y));
    __threadfence();
    __syncwarp();
    if (lane == 0) last = sk_ticket(ctr, nparts) ? 1 : 0;
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    if (!last) return false;
  }
  __syncwarp();
  __threadfence();
  if (nparts == 2) {  // one other part: p_lo + p_hi in either order, two chunks per batch of loads
    const int64_t c = me == c_lo ? c_hi : c_lo;
    const float4* src = sk_slot(p, c, sk_begin(sch, c) >= u_lo, w, lane);
#pragma unroll
    for (int kk = 0; kk < 4; kk += 2) {
      float4 v0[2][4], v1[2][4];
      sk_load8(src, kk, v0);
      sk_load8(src, kk + 1, v1);
      sk_add8(acc[kk], v0);
      sk_add8(acc[kk + 1], v1);
    }
    return true;
  }
  // three or more parts: this CTA's own in registers when it comes first, else
  // re-read with the rest (it was deposited: the shortcut above is taken only when
  // the own part can stay in registers)
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    float4 v0[2][4];
    if (me != c_lo) {
      sk_load8(sk_slot(p, c_lo, sk_begin(sch, c_lo) >= u_lo, w, lane), kk, v0);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          acc[kk][hf][x][0] = make_float2(v0[hf][x].x, v0[hf][x].y);
          acc[kk][hf][x][1] = make_float2(v0[hf][x].z, v0[hf][x].w);
        }
    }
    for (int64_t c = c_lo + 1; c <= c_hi; ++c) {
      sk_load8(sk_slot(p, c, sk_begin(sch, c) >= u_lo, w, lane), kk, v0);
      sk_add8(acc[kk], v0);
    }
  }
  return true;
}

// ------------------------------------------------------------------ roles
template <class SM>
__device__ __forceinline__ void load_weights(const GArgs& p, SM& S, const CUtensorMap* wmap, const Tile& T, int s,
                                             int slot) {
  uint8_t* wst = S.raw[slot] + T.cw * SM::AROW;
  for (int i = 0; i < T.g; ++i) {
    if constexpr (SM::WX) {  // pre-expanded weights: 128 rows x 128 bytes, 128-byte swizzle
      tma_2d(wst, wmap, s * KB * 32, static_cast<int32_t>(T.wrow0 + i * TW), &S.full_raw[slot]);
    } else {  // codes: 128 rows x 64 bytes, 64-byte swizzle
      tma_2d(wst + i * SM::WSUB, wmap, s * KB * 16, static_cast<int32_t>(T.wrow0 + i * TW), &S.full_raw[slot]);
    }
  }
}
template <class SM>
__device__ __forceinline__ void load_acts(const GArgs& p, SM& S, const CUtensorMap* amap, const Tile& T, int s,
                                          int slot) {
  uint8_t* st = S.raw[slot];
  for (int j = 0; j < T.cw / 32; ++j) {
    if constexpr (SM::AX) {  // expanded: 32 rows x 128 bytes, 128-byte swizzle
      tma_2d(st + j * 4096, amap, s * KB * 32, static_cast<int32_t>(T.a_row0) + 32 * j, &S.full_raw[slot]);
    } else {  // codes: 32 rows x 64 bytes
      tma_2d(st + j * 2048, amap, s * KB * 16, static_cast<int32_t>(T.a_row0) + 32 * j, &S.full_raw[slot]);
    }
  }
}

template <class SM>
__device__ void producer(const GArgs& p, SM& S, const CUtensorMap* wmap, const CUtensorMap* amap) {
  const int64_t B = p.K / 32;
  const int nst = static_cast<int>((B + KB - 1) / KB);
  if (p.producer_delay_ns) {  // test hook: hold the first copies back (bounded by the delay itself)
    const uint64_t t0 = gtime();
    while (!S.abort && gtime() - t0 < p.producer_delay_ns) {
    }
  }
  uint32_t gstage = 0;
  int64_t next = 0;
  Seg sg;
  bool have = false;
  Sched sch{};
  // The dense work list needs nothing from the previous kernel: the first stages'
  // weight copies go out before waiting for it (their slots are free on entry),
  // so that they overlap the kernel that writes the activations.
  int pre = 0;
  if (!p.segs) {
    sch = make_sched(p, nst);
    next = seg_start(sch);
    have = seg_next(sch, nst, next, sg);
    if (have && !S.abort) {
      const Tile T = tile_at(p, sg.t);
      const uint32_t bytes = static_cast<uint32_t>(T.cw * SM::AROW + T.g * SM::WSUB);
      for (; pre < RAW && sg.s0 + pre < sg.s1; ++pre) {
        mbar_expect_tx(&S.full_raw[pre], bytes);
        load_weights(p, S, wmap, T, sg.s0 + pre, pre);
      }
    }
  }
  grid_dep_wait();
  int skip = 0;  // stages of the first segment already issued
  if (pre > 0) {  // their activation copies, always, so that their stages complete
    const Tile T = tile_at(p, sg.t);
    for (int j = 0; j < pre; ++j) load_acts(p, S, amap, T, sg.s0 + j, j);
    gstage = pre;
    skip = pre;
  }
  if (p.segs) {
    sch = make_sched(p, nst);
    next = seg_start(sch);
    have = seg_next(sch, nst, next, sg);
  }
  bool stop = false;
  while (have && !stop && !S.abort) {
    const Tile T = tile_at(p, sg.t);
    const uint32_t bytes = static_cast<uint32_t>(T.cw * SM::AROW + T.g * SM::WSUB);
    for (int s = sg.s0 + skip; s < sg.s1; ++s) {
      const int slot = gstage % RAW;
      if (!bwait(&S.empty_raw[slot], ((gstage / RAW) & 1) ^ 1, S, p)) {
        stop = true;
        break;
      }
      mbar_expect_tx(&S.full_raw[slot], bytes);
      load_weights(p, S, wmap, T, s, slot);
      load_acts(p, S, amap, T, s, slot);
      ++gstage;
    }
    skip = 0;
    if (!stop) have = seg_next(sch, nst, next, sg);
  }
  // the copies in flight must land before the CTA exits
  const uint32_t first = gstage > RAW ? gstage - RAW : 0;
  for (uint32_t g = first; g < gstage; ++g) {
    const uint64_t t0 = gtime();
    while (!mbar_try(&S.full_raw[g % RAW], (g / RAW) & 1) && gtime() - t0 < kDrainNs) {
    }
  }
}

template <class SM>
__device__ void mma_issuer(const GArgs& p, SM& S, uint32_t tmem) {
  constexpr bool WX = SM::WX;
  const int64_t B = p.K / 32;
  const int nst = static_cast<int>((B + KB - 1) / KB);
  grid_dep_wait();
  const Sched sch = make_sched(p, nst);
  uint32_t gblk = 0, gst = 0;
  int64_t next = seg_start(sch);
  Seg sg;
  while (seg_next(sch, nst, next, sg)) {
    const Tile T = tile_at(p, sg.t);
    const uint32_t idesc = f8_idesc(T.cw);
    for (int s = sg.s0; s < sg.s1; ++s, ++gst) {
      const int slot = gst % RAW;
      const int nbk = static_cast<int>(B - static_cast<int64_t>(s) * KB < KB ? B - static_cast<int64_t>(s) * KB : KB);
      if (!bspin(&S.full_raw[slot], (gst / RAW) & 1, S, p)) goto done;
      const uint8_t* st = S.raw[slot];
      for (int kb = 0; kb < nbk; ++kb, ++gblk) {
        const int f = gblk % SM::F8;
        const int tb = gblk % NBUF;
        if (!WX && !bspin(&S.f8_full[f], (gblk / SM::F8) & 1, S, p)) goto done;
        if (!bspin(&S.tm_empty[tb], ((gblk / NBUF) & 1) ^ 1, S, p)) goto done;
        tc_fence_after();
        // activations: block kb of the raw stage (bytes 32kb.. of each swizzled 128-byte
        // row) or the converted operand next to the weights (8-row groups 256 bytes apart)
        const uint64_t bdesc = SM::AX ? kmajor_desc_sw128(st + kb * 32) : kmajor_desc(S.f8[f] + SM::F8W);
        for (int i = 0; i < T.g; ++i) {
          const uint64_t adesc = WX ? kmajor_desc_sw128(st + T.cw * SM::AROW + kb * 32)
                                    : kmajor_desc(S.f8[f] + i * 4096);
          mma_f8(tmem + static_cast<uint32_t>(tb * TCOLS + i * T.cw), adesc, bdesc, idesc);
        }
        mma_commit(&S.tm_full[tb]);
        if (!WX) mma_commit(&S.f8_empty[f]);
        if (kb == nbk - 1) mma_commit(&S.empty_raw[slot]);  // the stage's operands are read
      }
    }
  }
done:
  mma_commit(&S.mma_done);  // every MMA issued so far completes before TMEM is released
  const uint64_t t0 = gtime();
  while (!mbar_try(&S.mma_done, 0) && gtime() - t0 < kDrainNs) {
  }
}

// Four scales of one row (blocks 4s .. 4s + 3, clamped; validity applied later).
__device__ __forceinline__ uint4 ld_f4(const float* row, int s, int B, bool vec) {
  if (vec) return __ldg(reinterpret_cast<const uint4*>(row + s * KB));
  uint32_t v[KB];
#pragma unroll
  for (int k = 0; k < KB; ++k) v[k] = __float_as_uint(__ldg(row + min(s * KB + k, B - 1)));
  return make_uint4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ uint2 ld_h4(const uint16_t* row, int s, int B, bool vec) {
  if (vec) return __ldg(reinterpret_cast<const uint2*>(row + s * KB));
  uint32_t v[KB];
#pragma unroll
  for (int k = 0; k < KB; ++k) v[k] = __ldg(row + min(s * KB + k, B - 1));
  return make_uint2(v[0] | (v[1] << 16), v[2] | (v[3] << 16));
}

// One stage's scales into scale slot sc, by the helper threads (t of HT), in two
// phases of loads issued together (one round trip to L2 each): d_a per column,
// then d_w 2^18 and -d_w 8 S_w per weight row, stored in the orders the workers
// read.
template <class SM, int HT>
__device__ __forceinline__ void publish_scales(const GArgs& p, SM& S, const Tile& T, int s, int sc, int t, bool vec) {
  constexpr int AR = (TCOLS + HT - 1) / HT;          // columns per helper thread
  constexpr int WR = (SM::F8W / 32 + HT - 1) / HT;   // weight rows per helper thread
  const int64_t B64 = p.K / 32;
  const int B = static_cast<int>(B64);
  const int nbk = min(KB, B - s * KB);
  const int cols = T.g * T.cw;
  {
    uint4 av[AR];
#pragma unroll
    for (int i = 0; i < AR; ++i) {
      const int c = min(t + HT * i, TCOLS - 1);
      const int si = SM::G == 1 ? 0 : c / T.cw, jt = c - si * T.cw;
      const bool ok = c < cols && jt < T.ntok;
      av[i] = ld_f4(p.a_scales + (T.a_row0 + (ok ? jt : 0)) * B64, s, B, vec);
    }
#pragma unroll
    for (int i = 0; i < AR; ++i) {
      const int c = t + HT * i;
      if (c < TCOLS) {
        const int si = SM::G == 1 ? 0 : c / T.cw, jt = c - si * T.cw;
        const bool ok = c < cols && jt < T.ntok;
        const uint32_t w4[KB] = {av[i].x, av[i].y, av[i].z, av[i].w};
        const int cs = col_slot(c);
#pragma unroll
        for (int kk = 0; kk < KB; ++kk) S.sda[sc][kk][cs] = (ok && kk < nbk) ? __uint_as_float(w4[kk]) : 0.f;
      }
    }
  }
  // weight rows in batches of at most 4 per thread (the loads of a batch go out together)
  constexpr int RB = WR < 4 ? WR : 4;
#pragma unroll
  for (int i0 = 0; i0 < WR; i0 += RB) {
    uint2 dh[RB], sw[RB];
#pragma unroll
    for (int i = 0; i < RB; ++i) {
      const int r = min(t + HT * (i0 + i), SM::F8W / 32 - 1);
      const int si = r / TW, rr = r - si * TW;
      const bool ok = si < T.g && T.n0 + si * TW + rr < p.N;
      const int64_t row = T.wrow0 + (ok ? si * TW + rr : 0);
      dh[i] = ld_h4(p.w_scales + row * B64, s, B, vec);
      sw[i] = ld_h4(reinterpret_cast<const uint16_t*>(p.w_sums) + row * B64, s, B, vec);
    }
#pragma unroll
    for (int i = 0; i < RB; ++i) {
      const int r = t + HT * (i0 + i);
      if (i0 + i < WR && r < SM::F8W / 32) {
        const int si = r / TW, rr = r - si * TW;
        const bool ok = si < T.g && T.n0 + si * TW + rr < p.N;
        const int rs = row_slot(rr);
#pragma unroll
        for (int kk = 0; kk < KB; ++kk) {
          const uint32_t hw = kk < 2 ? dh[i].x : dh[i].y, sw2 = kk < 2 ? sw[i].x : sw[i].y;
          const bool v = ok && kk < nbk;
          const float dw =
              v ? __half2float(__ushort_as_half(static_cast<unsigned short>(hw >> (16 * (kk & 1))))) * fp8_unscale()
                : 0.f;
          const short sws = static_cast<short>(sw2 >> (16 * (kk & 1)));
          S.sdw[sc][kk][si][rs] = dw;
          // -d_w * 8 S_w, exact: (d_w 2^18) * (S_w 2^-15), at most 20 significant bits
          S.scorr[sc][kk][si][rs] = v ? -dw * (static_cast<float>(sws) * 3.0517578125e-05f) : 0.f;
        }
      }
    }
  }
}

// The helper warps, in two roles that run side by side.  Publishers (warps 2-3),
// stage by stage: once the workers have freed the scale slot, the stage's scale
// loads go out together (one round trip to L2) and the scales are published; the
// scale slots (4, or 2 in the G = 4 instance) let them run ahead of the fold.
// Converters (warps 12-15; none with pre-expanded weights), block by block: the
// stage's operand codes into an operand slot (8, or 3) ahead of the MMA.  Apart,
// the publishers' load latency does not hold up the conversion.
template <class SM>
__device__ void publishers(const GArgs& p, SM& S, int t) {
  constexpr int HT = 32 * SM::PUB;
  const int lane = threadIdx.x & 31;
  const int B = static_cast<int>(p.K / 32);
  const int nst = (B + KB - 1) / KB;
  const bool vec = (B % KB) == 0 && (reinterpret_cast<uintptr_t>(p.a_scales) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(p.w_scales) & 7) == 0 &&
                   (reinterpret_cast<uintptr_t>(p.w_sums) & 7) == 0;
  grid_dep_wait();
  const Sched sch = make_sched(p, nst);
  uint32_t gst = 0;
  int64_t next = seg_start(sch);
  Seg sg;
  while (seg_next(sch, nst, next, sg)) {
    const Tile T = tile_at(p, sg.t);
    for (int s = sg.s0; s < sg.s1; ++s, ++gst) {
      const int sc = gst % SM::NSC;
      if (!bwait(&S.sc_free[sc], ((gst / SM::NSC) & 1) ^ 1, S, p)) return;
      publish_scales<SM, HT>(p, S, T, s, sc, t, vec);
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.sc_ready[sc]);
    }
  }
}

template <class SM>
__device__ void converters(const GArgs& p, SM& S, int t) {
  constexpr int HT = 32 * SM::CONV;
  const int lane = threadIdx.x & 31;
  const int B = static_cast<int>(p.K / 32);
  const int nst = (B + KB - 1) / KB;
  grid_dep_wait();
  const Sched sch = make_sched(p, nst);
  uint32_t gst = 0, gblk = 0;
  int64_t next = seg_start(sch);
  Seg sg;
  while (seg_next(sch, nst, next, sg)) {
    const Tile T = tile_at(p, sg.t);
    for (int s = sg.s0; s < sg.s1; ++s, ++gst) {
      const int nbk = min(KB, B - s * KB);
      const int slot = gst % RAW;
      if (!bwait(&S.full_raw[slot], (gst / RAW) & 1, S, p)) return;
      const uint8_t* ast = S.raw[slot];
      const uint8_t* wst = ast + T.cw * SM::AROW;
      const int rows = T.g * TW;
      for (int kb = 0; kb < nbk; ++kb, ++gblk) {
        const int f = gblk % SM::F8;
        if (!bwait(&S.f8_empty[f], ((gblk / SM::F8) & 1) ^ 1, S, p)) return;
#pragma unroll 1
        for (int r = t; r < rows; r += HT) {
          const int si = r >> 7, rr = r & (TW - 1);
          // 64-byte swizzle of the TMA box: 16-byte chunk kb of row rr sits at kb ^ ((rr >> 1) & 3)
          const uint4 raw =
              *reinterpret_cast<const uint4*>(wst + si * SM::WSUB + rr * 64 + 16 * (kb ^ ((rr >> 1) & 3)));
          uint32_t l0, h0, l1, h1, l2, h2, l3, h3;
          q4_0_word_to_e4m3(raw.x, l0, h0);
          q4_0_word_to_e4m3(raw.y, l1, h1);
          q4_0_word_to_e4m3(raw.z, l2, h2);
          q4_0_word_to_e4m3(raw.w, l3, h3);
          uint8_t* d = S.f8[f] + si * 4096 + (rr >> 3) * 256 + (rr & 7) * 16;
          *reinterpret_cast<uint4*>(d) = make_uint4(l0, l1, l2, l3);        // elements 0-15
          *reinterpret_cast<uint4*>(d + 128) = make_uint4(h0, h1, h2, h3);  // elements 16-31
        }
        if constexpr (!SM::AX) {
          // activations: the offset codes a + 8 (nibble ^ 8) spread to bytes, the e4m3 operand
#pragma unroll 1
          for (int r = t; r < T.cw; r += HT) {
            const uint4 raw = *reinterpret_cast<const uint4*>(ast + r * 64 + 16 * kb);
            const uint32_t x0 = raw.x ^ 0x88888888u, x1 = raw.y ^ 0x88888888u;
            const uint32_t x2 = raw.z ^ 0x88888888u, x3 = raw.w ^ 0x88888888u;
            uint8_t* d = S.f8[f] + SM::F8W + (r >> 3) * 256 + (r & 7) * 16;
            *reinterpret_cast<uint4*>(d) =
                make_uint4(x0 & 0x0F0F0F0Fu, x1 & 0x0F0F0F0Fu, x2 & 0x0F0F0F0Fu, x3 & 0x0F0F0F0Fu);
            *reinterpret_cast<uint4*>(d + 128) = make_uint4((x0 >> 4) & 0x0F0F0F0Fu, (x1 >> 4) & 0x0F0F0F0Fu,
                                                            (x2 >> 4) & 0x0F0F0F0Fu, (x3 >> 4) & 0x0F0F0F0Fu);
          }
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.f8_full[f]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty_raw[slot]);  // the raw codes are converted
    }
  }
}

// The value index of a worker thread's accumulators: acc[kk][hf][x][s] holds rows
// 32q + 16hf + 8s + lane/4 (s < 2) and columns 32(h + 2kk) + 8x + 2(lane%4) + e.
struct FoldCtx {
  int q, h, jr, u, lane;
};

// The fold of one segment's blocks for a warp with NK chunks (0..4) in the tile:
// straight-line, every piece (chunk kk, 16-lane half hf) a 16x256b load of 16
// registers, the next piece's load in flight while the current one is folded.
// si[kk]: the weight sub-tile of chunk kk.  False if a wait gave up.
template <int NK, class SM>
__device__ __forceinline__ bool fold_segment(const GArgs& p, SM& S, uint32_t tmem, const FoldCtx& c,
                                             const int (&si)[4], int b0, int b_end, uint32_t gst0, uint32_t& gfold,
                                             float2 (&acc)[4][2][4][2]) {
  constexpr int NP = 2 * NK;
  for (int b = b0; b < b_end; ++b) {
    const int s = b / KB, kb = b - s * KB;
    const uint32_t gs = gst0 + static_cast<uint32_t>(s - b0 / KB);
    const int sc = gs % SM::NSC;
    if (kb == 0 && !bwait(&S.sc_ready[sc], (gs / SM::NSC) & 1, S, p)) return false;
    const int tb = gfold % NBUF;
    if (!bwait(&S.tm_full[tb], (gfold / NBUF) & 1, S, p)) return false;
    tc_fence_after();
    const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * c.q) << 16) + static_cast<uint32_t>(tb * TCOLS);
    if constexpr (NP > 0) {
      uint32_t ra[16], rb[16];
      tmem_ld16x256_x4(tbase + static_cast<uint32_t>(32 * c.h), ra);
      float4 dwv = *reinterpret_cast<const float4*>(&S.sdw[sc][kb][si[0]][32 * c.q + 4 * c.jr]);
      float4 crv = *reinterpret_cast<const float4*>(&S.scorr[sc][kb][si[0]][32 * c.q + 4 * c.jr]);
      float4 da0, da1;
      tmem_wait(ra);
#pragma unroll
      for (int pc = 0; pc < NP; ++pc) {
        const int kk = pc >> 1, hf = pc & 1;
        uint32_t(&cur)[16] = (pc & 1) ? rb : ra;
        uint32_t(&nxt)[16] = (pc & 1) ? ra : rb;
        if (pc + 1 < NP) {
          const int k1 = c.h + 2 * ((pc + 1) >> 1), hf1 = (pc + 1) & 1;
          tmem_ld16x256_x4(tbase + (static_cast<uint32_t>(16 * hf1) << 16) + static_cast<uint32_t>(32 * k1), nxt);
        }
        if (hf == 0) {
          if (SM::G > 1 && kk > 0 && si[kk] != si[kk - 1]) {  // a new weight sub-tile: its 4 rows' d_w, correction
            dwv = *reinterpret_cast<const float4*>(&S.sdw[sc][kb][si[kk]][32 * c.q + 4 * c.jr]);
            crv = *reinterpret_cast<const float4*>(&S.scorr[sc][kb][si[kk]][32 * c.q + 4 * c.jr]);
          }
          const float4* dap = reinterpret_cast<const float4*>(&S.sda[sc][kb][32 * (c.h + 2 * kk) + 8 * c.u]);
          da0 = dap[0];
          da1 = dap[1];
        }
        const float dA = hf ? dwv.z : dwv.x, dB = hf ? dwv.w : dwv.y;
        const float cA = hf ? crv.z : crv.x, cB = hf ? crv.w : crv.y;
        const float2 dw0 = make_float2(dA, dA), dw1 = make_float2(dB, dB);
        const float2 c0 = make_float2(cA, cA), c1 = make_float2(cB, cB);
        const float2 dav[4] = {make_float2(da0.x, da0.y), make_float2(da0.z, da0.w), make_float2(da1.x, da1.y),
                               make_float2(da1.z, da1.w)};
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const float2 t0 =
              __ffma2_rn(make_float2(__uint_as_float(cur[4 * x]), __uint_as_float(cur[4 * x + 1])), dw0, c0);
          const float2 t1 =
              __ffma2_rn(make_float2(__uint_as_float(cur[4 * x + 2]), __uint_as_float(cur[4 * x + 3])), dw1, c1);
          acc[kk][hf][x][0] = __ffma2_rn(t0, dav[x], acc[kk][hf][x][0]);
          acc[kk][hf][x][1] = __ffma2_rn(t1, dav[x], acc[kk][hf][x][1]);
        }
        if (pc + 1 < NP) {
          tmem_wait(nxt);
          if (pc + 2 == NP) {  // every piece of this block is in registers: the buffer goes back
            tc_fence_before();
            __syncwarp();
            if (c.lane == 0) mbar_arrive(&S.tm_empty[tb]);
          }
        }
      }
    } else {  // no chunk in this tile: hand the buffer back at once
      tc_fence_before();
      __syncwarp();
      if (c.lane == 0) mbar_arrive(&S.tm_empty[tb]);
    }
    if (kb == KB - 1 || b == b_end - 1) {  // this stage's scale slot is no longer read
      __syncwarp();
      if (c.lane == 0) mbar_arrive(&S.sc_free[sc]);
    }
    ++gfold;
  }
  return true;
}

// The single-weight-tile instance's output: per chunk kk and 8-token group x, the
// warp's 8 tokens x 32 features go through shared memory (a 1 KB staging buffer
// per warp) so that each lane stores two 16-byte runs of 4 features of one token
// row instead of eight 4-byte values; 16-byte groups are XOR-swizzled by token so
// that neither side conflicts on banks.  Rows past the segment's tokens and
// features past N are not written; unaligned Y falls back to 4-byte stores.
__device__ __forceinline__ void store_rows(const GArgs& p, float* ys, const Tile& T, const float2 (&acc)[4][2][4][2],
                                           int nk, int h, int q, int jr, int u, int lane) {
  const bool vec = (reinterpret_cast<uintptr_t>(p.y) & 15) == 0 && (p.ldy & 3) == 0;
  const int tr = lane >> 2;  // the token this lane stores
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    if (kk >= nk) continue;
    const int k = h + 2 * kk;
#pragma unroll
    for (int x = 0; x < 4; ++x) {
#pragma unroll
      for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int r = 0; r < 4; ++r) {  // token 2u + e, feature 8r + jr of the warp's 32
          const int t = 2 * u + e, f = 8 * r + jr;
          const float2 a2 = acc[kk][r >> 1][x][r & 1];
          ys[t * 32 + 4 * ((f >> 2) ^ t) + (f & 3)] = e ? a2.y : a2.x;
        }
      __syncwarp();
      const int jt = 32 * k + 8 * x + tr;  // token within the segment
      if (jt < T.ntok) {
        const int64_t orow = p.perm ? static_cast<int64_t>(p.perm[T.a_row0 + jt]) : T.a_row0 + jt;
        float* yr = p.y + orow * p.ldy;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          const int f4 = 2 * (lane & 3) + g;
          const float4 v = *reinterpret_cast<const float4*>(&ys[tr * 32 + 4 * (f4 ^ tr)]);
          const int64_t n = T.n0 + 32 * q + 4 * f4;
          if (vec && n + 3 < p.N) {
            *reinterpret_cast<float4*>(yr + n) = v;
          } else {
            if (n < p.N) yr[n] = v.x;
            if (n + 1 < p.N) yr[n + 1] = v.y;
            if (n + 2 < p.N) yr[n + 2] = v.z;
            if (n + 3 < p.N) yr[n + 3] = v.w;
          }
        }
      }
      __syncwarp();
    }
  }
}

template <class SM>
__device__ void workers(const GArgs& p, SM& S, uint32_t tmem) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;  // 4..11
  FoldCtx c;
  c.q = warp & 3;                // TMEM lane quarter
  c.h = (warp - 4) >> 2;         // chunk parity: chunks h, h + 2, h + 4, h + 6
  c.jr = lane >> 2;
  c.u = lane & 3;
  c.lane = lane;
  const int q = c.q, h = c.h, jr = c.jr, u = c.u;
  const int64_t B64 = p.K / 32;
  const int B = static_cast<int>(B64);
  const int nst = (B + KB - 1) / KB;
  grid_dep_wait();
  const Sched sch = make_sched(p, nst);
  uint32_t gfold = 0, gst = 0;
  int64_t next = seg_start(sch);
  Seg sg;
  while (seg_next(sch, nst, next, sg)) {
    const Tile T = tile_at(p, sg.t);
    const int nch = T.g * T.cw / 32;                  // 32-column chunks in the tile
    const int nk = nch > h ? (nch - h + 1) / 2 : 0;   // this warp's chunks
    int si[4];  // weight sub-tile of each of this warp's chunks
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) si[kk] = SM::G == 1 ? 0 : min((32 * (h + 2 * kk)) / T.cw, T.g - 1);
    float2 acc[4][2][4][2];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          acc[a][b][x][0] = make_float2(0.f, 0.f);
          acc[a][b][x][1] = make_float2(0.f, 0.f);
        }
    const int b0 = sg.s0 * KB, b_end = min(sg.s1 * KB, B);
    bool ok;
    switch (nk) {
      case 4: ok = fold_segment<4>(p, S, tmem, c, si, b0, b_end, gst, gfold, acc); break;
      case 3: ok = fold_segment<3>(p, S, tmem, c, si, b0, b_end, gst, gfold, acc); break;
      case 2: ok = fold_segment<2>(p, S, tmem, c, si, b0, b_end, gst, gfold, acc); break;
      case 1: ok = fold_segment<1>(p, S, tmem, c, si, b0, b_end, gst, gfold, acc); break;
      default: ok = fold_segment<0>(p, S, tmem, c, si, b0, b_end, gst, gfold, acc); break;
    }
    if (!ok) return;
    gst += static_cast<uint32_t>(sg.s1 - sg.s0);

    // ---- epilogue
    const bool split = sch.U && (sg.s0 > 0 || sg.s1 < nst);
    if (split && !sk_epilogue(p, sch, sg, nst, warp - 4, lane, acc)) continue;
    if constexpr (SM::G == 1) {
      store_rows(p, S.ystage[warp - 4], T, acc, nk, h, q, jr, u, lane);
      continue;
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      if (kk >= nk) continue;
      const int k = h + 2 * kk;
      const int64_t nrow0 = T.n0 + si[kk] * TW;  // first output feature of the chunk's sub-tile
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int jt = 32 * k + 8 * x + 2 * u + e - si[kk] * T.cw;  // token within the segment
          if (jt >= T.ntok) continue;
          const int64_t orow = p.perm ? static_cast<int64_t>(p.perm[T.a_row0 + jt]) : T.a_row0 + jt;
          float* yr = p.y + orow * p.ldy;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf)
#pragma unroll
            for (int s2 = 0; s2 < 2; ++s2) {
              const int64_t n = nrow0 + 32 * q + 16 * hf + 8 * s2 + jr;
              if (n < p.N && n < nrow0 + TW) {
                const float2 a2 = acc[kk][hf][x][s2];
                yr[n] = e ? a2.y : a2.x;
              }
            }
        }
    }
  }
}

template <int G, bool WEXP, bool AEXP>
__global__ void __launch_bounds__(GSmem<G, WEXP, AEXP>::THREADS, 1)
    w4a4_grp_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap amap,
                    const GArgs p) {
  using SM = GSmem<G, WEXP, AEXP>;
  extern __shared__ __align__(1024) uint8_t smem_dyn[];
  SM& S = *reinterpret_cast<SM*>(smem_dyn);
  const int warp = threadIdx.x >> 5;
  if ((static_cast<uint32_t>(__cvta_generic_to_shared(smem_dyn)) & 1023u) != 0) {  // never expected
    if (threadIdx.x == 0) atomicOr(p.err, 2);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < RAW; ++i) {
      mbar_init(&S.full_raw[i], 1);
      // the converters' arrivals once the codes are converted, and the MMA's commit
      mbar_init(&S.empty_raw[i], SM::CONV + 1);
    }
    if constexpr (!WEXP) {  // (pre-expanded weights: no operand slots in use)
      for (int i = 0; i < SM::F8; ++i) {
        mbar_init(&S.f8_full[i], SM::CONV);
        mbar_init(&S.f8_empty[i], 1);
      }
    }
    for (int i = 0; i < NBUF; ++i) {
      mbar_init(&S.tm_full[i], 1);
      mbar_init(&S.tm_empty[i], kWorkers);
    }
    for (int i = 0; i < SM::NSC; ++i) {
      mbar_init(&S.sc_ready[i], SM::PUB);
      mbar_init(&S.sc_free[i], kWorkers);
    }
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
  // the next kernel on the stream may start its own set-up now
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const uint32_t tmem = S.tmem_base;
  if (warp < 4 || warp >= 12) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(SM::REGS_LOW));
    if (warp == 0) {
      if ((threadIdx.x & 31) == 0) producer(p, S, &wmap, &amap);
      __syncwarp();
    } else if (warp == 1) {
      if ((threadIdx.x & 31) == 0) mma_issuer(p, S, tmem);
      __syncwarp();
    } else if (warp < 4) {  // publishers: warps 2-3
      publishers(p, S, threadIdx.x - 64);
    } else {  // converters: warps 12-15
      converters(p, S, threadIdx.x - 384);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(SM::REGS_HIGH));
    workers(p, S, tmem);
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
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// Q4_0 codes [rows][K/2]: box 64 bytes x 128 rows, 64-byte swizzle.
cudaError_t codes_map_sw64(CUtensorMap* m, const uint8_t* codes, int64_t rows, int64_t K) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(KB * 16), static_cast<cuuint32_t>(TW)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(codes), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Expanded operand bytes [rows][K]: box 128 bytes (one stage of 4 blocks) x
// box_rows rows, 128-byte swizzle (the MMA's K-major swizzled layout).  Rows past
// `rows` read as zero.
cudaError_t expanded_map_sw128(CUtensorMap* m, const uint8_t* x, int64_t rows, int64_t K, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(KB * 32), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(x), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

std::mutex g_cfg_mu;

template <int G, bool WEXP, bool AEXP>
cudaError_t launch_grp(const CUtensorMap& wmap, const CUtensorMap& amap, const GArgs& a, int grid,
                       cudaStream_t stream) {
  auto kern = w4a4_grp_kernel<G, WEXP, AEXP>;
  using SM = GSmem<G, WEXP, AEXP>;
  constexpr size_t kSmem = sizeof(SM);
  static bool configured[64] = {};
  static int regs_ok[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(g_cfg_mu);
    if (!configured[dev]) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmem));
      if (e != cudaSuccess) return e;
      // setmaxnreg.inc waits until the block's launch registers cover the split:
      // refuse a build whose register count would make it wait forever
      cudaFuncAttributes fa{};
      e = cudaFuncGetAttributes(&fa, kern);
      if (e != cudaSuccess) return e;
      regs_ok[dev] = (fa.numRegs * SM::THREADS >= (SM::THREADS - 256) * SM::REGS_LOW + 256 * SM::REGS_HIGH) ? 1 : -1;
      configured[dev] = true;
    }
  }
  if (regs_ok[dev] < 0) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(SM::THREADS);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, wmap, amap, a);
}

// Stream-K plan of the dense product (as for gemm_tc.cu): used where it shortens
// the longest CTA by more than 10% (a fix-up counted as two stages).
constexpr int64_t kSkMaxTiles = 32768;
constexpr size_t kSkTicketBytes = static_cast<size_t>(kSkMaxTiles) * 8 * sizeof(uint32_t);  // 1 MiB
constexpr size_t kSkPartBytes = size_t(8) * 1024 * sizeof(float4);

struct GPlan {
  int g;           // weight tiles per tile
  int64_t nseg;    // token segments
  int64_t tiles;
  bool sk;
  int64_t units;
  int grid;
  size_t ws_bytes;
};

GPlan plan_dense(int64_t M, int64_t N, int64_t K, bool allow_multi) {
  GPlan pl{};
  if (M <= 0 || N <= 0 || K <= 0) return pl;
  const int64_t NT = (N + TW - 1) / TW;
  pl.nseg = (M + TCOLS - 1) / TCOLS;
  const int64_t cw = pl.nseg == 1 ? ((M + 31) & ~int64_t(31)) : TCOLS;
  pl.g = allow_multi ? static_cast<int>(std::min<int64_t>({4, TCOLS / cw, NT})) : 1;
  if (pl.g > 1) {  // balanced groups of weight tiles
    const int64_t ng = (NT + pl.g - 1) / pl.g;
    pl.g = static_cast<int>((NT + ng - 1) / ng);
  }
  pl.tiles = pl.nseg * ((NT + pl.g - 1) / pl.g);
  const int64_t nst = (K / 32 + KB - 1) / KB;
  const int64_t sms = num_sms();
  pl.grid = static_cast<int>(pl.tiles < sms ? pl.tiles : sms);
  const int64_t dp_span = ((pl.tiles + sms - 1) / sms) * nst;
  const int64_t U = pl.tiles * nst;
  const int64_t Gr = U < sms ? U : sms;
  const int64_t sk_span = (U + Gr - 1) / Gr + 2;
  if (Gr >= 2 && pl.tiles <= kSkMaxTiles && 10 * sk_span < 9 * dp_span) {
    pl.sk = true;
    pl.units = U;
    pl.grid = static_cast<int>(Gr);
    pl.ws_bytes = kSkTicketBytes + 2 * static_cast<size_t>(Gr) * kSkPartBytes;
  }
  return pl;
}

// Test hooks (w4a4_debug_set_wait_limit): the pipeline-wait bound and the producer delay.
uint64_t g_wait_ns = 1000000000ull;
uint64_t g_delay_ns = 0;

}  // namespace

void grp_set_wait_limit(uint64_t wait_ns, uint64_t producer_delay_ns) {
  g_wait_ns = wait_ns ? wait_ns : 1000000000ull;
  g_delay_ns = producer_delay_ns;
}

size_t grp_sk_part_bytes() { return kSkPartBytes; }

size_t grp_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  const GPlan pl = plan_dense(M, N, K, M <= TCOLS);
  return pl.sk ? pl.ws_bytes : 0;
}

cudaError_t launch_gemm_grp(const uint8_t* w_codes, const uint16_t* w_scales, const int16_t* w_sums,
                            const uint8_t* w_expanded, int64_t N, const uint8_t* a_expanded, const float* a_scales,
                            int64_t M, int64_t K, float* y, int64_t ldy, void* ws, size_t ws_bytes,
                            cudaStream_t stream) {
  const bool small = M <= TCOLS;  // one token segment: several weight tiles per tile
  const GPlan pl = plan_dense(M, N, K, small);
  GArgs a{};
  a.w_scales = w_scales; a.w_sums = w_sums; a.a_scales = a_scales;
  a.y = y; a.ldy = ldy; a.M = M; a.N = N; a.K = K;
  a.NT = static_cast<int>((N + TW - 1) / TW);
  a.dense_g = pl.g;
  a.dense_nseg = pl.nseg;
  a.err = device_error_word();
  if (!a.err) return cudaErrorInvalidSymbol;
  a.wait_ns = g_wait_ns;
  a.producer_delay_ns = g_delay_ns;
  int grid = pl.grid;
  if (pl.sk && ws && ws_bytes >= pl.ws_bytes) {
    a.sk_units = pl.units;
    a.sk_count = static_cast<uint32_t*>(ws);
    a.sk_part = reinterpret_cast<float4*>(static_cast<uint8_t*>(ws) + kSkTicketBytes);
  } else {
    grid = static_cast<int>(std::min<int64_t>(pl.tiles, num_sms()));
  }
  const bool wexp = w_expanded != nullptr && pl.g == 1;
  CUtensorMap wmap, amap;
  cudaError_t e = wexp ? expanded_map_sw128(&wmap, w_expanded, N, K, TW) : codes_map_sw64(&wmap, w_codes, N, K);
  if (e == cudaSuccess) e = expanded_map_sw128(&amap, a_expanded, M, K, 32);
  if (e != cudaSuccess) return e;
  if (pl.g > 1) return launch_grp<4, false, true>(wmap, amap, a, grid, stream);
  if (wexp) return launch_grp<1, true, true>(wmap, amap, a, grid, stream);
  return launch_grp<1, false, true>(wmap, amap, a, grid, stream);
}

cudaError_t launch_gemm_grp_routed(const uint8_t* w_codes, const uint16_t* w_scales, const int16_t* w_sums,
                                   int E, int64_t N, int64_t K, const Routing& r, float* y,
                                   cudaStream_t stream) {
  GArgs a{};
  a.w_scales = w_scales; a.w_sums = w_sums; a.a_scales = r.gscales;
  a.y = y; a.ldy = N; a.M = 0; a.N = N; a.K = K;
  a.NT = static_cast<int>((N + TW - 1) / TW);
  a.dense_g = 1;
  a.segs = r.segs;
  a.seg_tiles = r.seg_tiles;
  a.counts = r.hdr + 1;
  a.perm = r.perm;
  a.err = device_error_word();
  if (!a.err) return cudaErrorInvalidSymbol;
  a.wait_ns = g_wait_ns;
  a.producer_delay_ns = g_delay_ns;
  // stream-K over the routing kernel's tiles: the units are counted on the device
  int grid = num_sms();
  if (r.sk_part && r.sk_count && r.sk_ctas > 0) {
    a.sk_dyn = 1;
    a.sk_count = r.sk_count;
    a.sk_part = r.sk_part;
    grid = r.sk_ctas;
  }
  CUtensorMap wmap, amap;
  cudaError_t e = codes_map_sw64(&wmap, w_codes, static_cast<int64_t>(E) * N, K);
  if (e == cudaSuccess)
    e = encode_2d_map(&amap, CU_TENSOR_MAP_DATA_TYPE_UINT8, r.gcodes, static_cast<uint64_t>(K / 2),
                      static_cast<uint64_t>(r.rows), static_cast<uint64_t>(K / 2), KB * 16, 32,
                      CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  return launch_grp<4, false, false>(wmap, amap, a, grid, stream);
}

}  // namespace w4a4
