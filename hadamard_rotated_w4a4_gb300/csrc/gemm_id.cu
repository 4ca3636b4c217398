// Expert-routed W4A4 product (MUL_MAT_ID), engine docs "The lean option:
// ROCmFP4, ROCmI4 and Hadamard Q4_0", section "MoE: W4A4 on the experts": the
// W4A4 kernel runs the expert matmuls too, where an MoE spends nearly all of its
// prompt work.
//
// Three launches on the caller's stream, each of the later two allowed to start
// while the one before finishes (programmatic dependent launch):
//   1. route (one CTA): the (token, slot) pairs per expert, their exclusive scan,
//      the pair list grouped by expert, and the GEMM's work list -- each expert's
//      rows cut into segments of at most 256, each segment paired with groups of
//      up to 4 weight tiles so that a tile fills up to 256 accumulator columns;
//      ids outside [0, E) zero their output row and set a device flag;
//   2. gather (every SM): each routed row's int4 codes and scales, copied in
//      expert order so that every segment is contiguous;
//   3. the super-tile GEMM (gemm_grp.cu) over the work list, scattering each
//      output row to its (token, slot).
#include <mutex>

#include "w4a4_kernels.cuh"

namespace w4a4 {

namespace {

constexpr int kRouteThreads = 1024;
constexpr int kSegRows = 256;  // token rows per segment (the GEMM's accumulator columns)
constexpr int kMaxG = 4;       // weight tiles per tile

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Weight tiles per tile of a segment of `ntok` rows, balanced over the NT tiles.
__device__ __forceinline__ int seg_group(int ntok, int NT) {
  const int cw = (ntok + 31) & ~31;
  const int gmax = min(min(kMaxG, kSegRows / cw), NT);
  const int ng = (NT + gmax - 1) / gmax;
  return (NT + ng - 1) / ng;
}

// Block-wide exclusive scan of one value per thread (kRouteThreads threads).
__device__ __forceinline__ int block_excl_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = lane < kRouteThreads / 32 ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, t, o);
      if (lane >= o) t += y;
    }
    warp_tot[lane] = t;  // inclusive over warps
    if (lane == 31) *total = t;
  }
  __syncthreads();
  const int before = (warp > 0 ? warp_tot[warp - 1] : 0) + x - v;
  __syncthreads();  // warp_tot is reused by the next scan
  return before;
}

__global__ void __launch_bounds__(kRouteThreads) route_kernel(const int32_t* __restrict__ ids, int64_t npairs,
                                                               int E, int64_t N, int NT, float* __restrict__ y,
                                                               Routing r) {
  extern __shared__ int32_t sh[];  // cnt[E], cursor[E]
  int32_t* cnt = sh;
  int32_t* cur = sh + E;
  __shared__ int warp_tot[32];
  __shared__ int tot[3];
  __shared__ int bad;
  grid_dep_launch();
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
  if (tid == 0) bad = 0;
  __syncthreads();
  for (int64_t i = tid; i < npairs; i += blockDim.x) {
    const int e = ids[i];
    if (e >= 0 && e < E) {
      atomicAdd(&cnt[e], 1);
    } else {
      bad = 1;
      float4* yr = reinterpret_cast<float4*>(y + i * N);  // an unused slot's output row is zero
      if ((N & 3) == 0 && (reinterpret_cast<uintptr_t>(y) & 15) == 0) {
        for (int64_t n = 0; n < N / 4; ++n) yr[n] = make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
        for (int64_t n = 0; n < N; ++n) y[i * N + n] = 0.f;
      }
    }
  }
  __syncthreads();
  // each thread owns a run of consecutive experts: its rows, segments and tiles
  const int per = (E + kRouteThreads - 1) / kRouteThreads;
  const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
  int rows = 0, segs = 0, tiles = 0;
  for (int e = e0; e < e1; ++e) {
    const int n = cnt[e];
    rows += n;
    for (int s = 0; s * kSegRows < n; ++s) {
      const int g = seg_group(min(kSegRows, n - s * kSegRows), NT);
      ++segs;
      tiles += (NT + g - 1) / g;
    }
  }
  int row0 = block_excl_scan(rows, warp_tot, &tot[0]);
  int seg0 = block_excl_scan(segs, warp_tot, &tot[1]);
  int tile0 = block_excl_scan(tiles, warp_tot, &tot[2]);
  for (int e = e0; e < e1; ++e) {
    const int n = cnt[e];
    r.offsets[e] = row0;
    cur[e] = row0;
    for (int s = 0; s * kSegRows < n; ++s) {
      const int ntok = min(kSegRows, n - s * kSegRows);
      const int g = seg_group(ntok, NT);
      r.segs[seg0] = make_int4(row0 + s * kSegRows, e, ntok, g);
      r.seg_tiles[seg0] = tile0;
      ++seg0;
      tile0 += (NT + g - 1) / g;
    }
    row0 += n;
  }
  if (tid == 0) {
    r.offsets[E] = tot[0];
    r.seg_tiles[tot[1]] = tot[2];
    r.hdr[0] = bad;
    r.hdr[1] = tot[1];  // segments
    r.hdr[2] = tot[2];  // tiles
    r.hdr[3] = tot[0];  // routed rows
  }
  __syncthreads();
  for (int64_t i = tid; i < npairs; i += blockDim.x) {
    const int e = ids[i];
    if (e >= 0 && e < E) r.perm[atomicAdd(&cur[e], 1)] = static_cast<int32_t>(i);
  }
  // the GEMM's stream-K tickets start at zero (they return to zero after each use;
  // clearing them here also recovers from a launch that gave up)
  if (r.sk_count)
    for (int i = tid; i < r.sk_ctas * 8; i += blockDim.x) r.sk_count[i] = 0u;
}

// One warp per routed row: its code bytes (16-byte chunks) and scales, in expert order.
__global__ void __launch_bounds__(256) gather_kernel(const uint8_t* __restrict__ codes,
                                                     const float* __restrict__ scales, int64_t K, int top_k,
                                                     int act_per_slot, Routing r) {
  grid_dep_wait();
  grid_dep_launch();
  const int64_t rows = r.hdr[3];
  const int64_t B = K / 32;
  const int lane = threadIdx.x & 31;
  const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t i = w0; i < rows; i += nw) {
    const int64_t pr = r.perm[i];
    const int64_t src = act_per_slot ? pr : pr / top_k;
    const uint4* s = reinterpret_cast<const uint4*>(codes + src * (K / 2));
    uint4* d = reinterpret_cast<uint4*>(r.gcodes + i * (K / 2));
    for (int64_t c = lane; c < B; c += 32) d[c] = s[c];
    const float* ss = scales + src * B;
    float* ds = r.gscales + i * B;
    for (int64_t c = lane; c < B; c += 32) ds[c] = ss[c];
  }
}

size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

}  // namespace

RoutingLayout routing_layout(int64_t npairs, int E, int64_t K) {
  RoutingLayout L{};
  const int64_t max_seg = (npairs + kSegRows - 1) / kSegRows + E;
  size_t off = 0;
  L.hdr = off;       off += 16;  // flag first, so that a status query needs only the pointer
  L.offsets = off;   off += align16(sizeof(int32_t) * static_cast<size_t>(E + 1));
  L.segs = off;      off += align16(16 * static_cast<size_t>(max_seg));
  L.seg_tiles = off; off += align16(sizeof(int32_t) * static_cast<size_t>(max_seg + 1));
  L.perm = off;      off += align16(sizeof(int32_t) * static_cast<size_t>(npairs));
  L.gcodes = off;    off += align16(static_cast<size_t>(npairs) * static_cast<size_t>(K / 2));
  L.gscales = off;   off += align16(static_cast<size_t>(npairs) * static_cast<size_t>(K / 32) * sizeof(float));
  // stream-K over the routed tiles: one ticket per (tile's first CTA, worker warp),
  // two partial tiles per CTA
  L.sk_ctas = num_sms();
  L.sk_count = off;  off += align16(sizeof(uint32_t) * 8 * static_cast<size_t>(L.sk_ctas));
  off = (off + 255) & ~size_t(255);
  L.sk_part = off;   off += 2 * static_cast<size_t>(L.sk_ctas) * grp_sk_part_bytes();
  L.total = off;
  return L;
}

Routing routing_in(void* ws, int64_t npairs, int E, int64_t K) {
  const RoutingLayout L = routing_layout(npairs, E, K);
  uint8_t* base = static_cast<uint8_t*>(ws);
  Routing r;
  r.hdr = reinterpret_cast<int32_t*>(base + L.hdr);
  r.offsets = reinterpret_cast<int32_t*>(base + L.offsets);
  r.segs = reinterpret_cast<int4*>(base + L.segs);
  r.seg_tiles = reinterpret_cast<int32_t*>(base + L.seg_tiles);
  r.perm = reinterpret_cast<int32_t*>(base + L.perm);
  r.gcodes = base + L.gcodes;
  r.gscales = reinterpret_cast<float*>(base + L.gscales);
  r.rows = npairs;
  r.sk_count = reinterpret_cast<uint32_t*>(base + L.sk_count);
  r.sk_part = reinterpret_cast<float4*>(base + L.sk_part);
  r.sk_ctas = L.sk_ctas;
  return r;
}

// One routing scratch per device, for callers without a workspace.  The
// kernels write every word they read, so it is never cleared.
static __device__ __align__(256) uint8_t g_id_scratch[kIdStaticScratchBytes];

cudaError_t id_static_scratch(void** addr) {
  static std::mutex mu;
  static void* cached[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_id_scratch);  // the current device's copy
    if (e != cudaSuccess) return e;
    if (!p) return cudaErrorInvalidSymbol;
    cached[dev] = p;
  }
  *addr = cached[dev];
  return cudaSuccess;
}

cudaError_t launch_gemm_id(const uint8_t* w_codes, const uint16_t* w_scales, const int16_t* w_sums, int E,
                           int64_t N, const uint8_t* a_codes, const float* a_scales, int64_t K, const int32_t* ids,
                           int64_t M, int top_k, int act_per_slot, float* y, const Routing& r, cudaStream_t stream) {
  const int64_t npairs = M * top_k;
  const int NT = static_cast<int>((N + 127) / 128);
  const size_t sh = sizeof(int32_t) * 2 * static_cast<size_t>(E);
  if (sh > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(sh));
    if (e != cudaSuccess) return e;
  }
  route_kernel<<<1, kRouteThreads, sh, stream>>>(ids, npairs, E, N, NT, y, r);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  const int64_t gwarps = npairs < 8 * 1024 ? npairs : 8 * 1024;
  cfg.gridDim = dim3(static_cast<unsigned>((gwarps + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, gather_kernel, a_codes, a_scales, K, top_k, act_per_slot, r);
  if (e != cudaSuccess) return e;
  return launch_gemm_grp_routed(w_codes, w_scales, w_sums, E, N, K, r, y, stream);
}

}  // namespace w4a4
