// Expert-routed W4A4 product (MUL_MAT_ID), engine docs "The lean option:
// ROCmFP4, ROCmI4 and Hadamard Q4_0", section "MoE: W4A4 on the experts": the
// W4A4 kernel runs the expert matmuls too, where an MoE spends nearly all of its
// prompt work.
//
// Three launches on the caller's stream:
//   1. route_prep (one CTA): histogram of ids per expert, exclusive scans of the
//      pair counts and of the row tiles per expert, the pair list grouped by
//      expert, zeroed output rows and a device flag for ids outside [0, E);
//   2. gather: each routed row's activation codes and scales, copied in expert
//      order into the workspace, so that every expert's rows are contiguous;
//   3. the grouped GEMM over (expert row tile, weight tile), loading both
//      operands with 2D TMA and scattering each output row to (token, slot).
#include <mutex>

#include "w4a4_kernels.cuh"

namespace w4a4 {

namespace {

constexpr int kPrepThreads = 1024;

__global__ void __launch_bounds__(kPrepThreads) route_prep_kernel(const int32_t* __restrict__ ids, int64_t npairs,
                                                                   int E, int64_t N, int tile_tokens,
                                                                   float* __restrict__ y, Routing r) {
  extern __shared__ int32_t sh[];  // cnt[E], cursor[E]
  int32_t* cnt = sh;
  int32_t* cur = sh + E;
  __shared__ int bad;
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
      float* yr = y + i * N;  // an unused slot's output row is zero
      for (int64_t n = 0; n < N; ++n) yr[n] = 0.f;
    }
  }
  __syncthreads();
  if (tid == 0) {
    int32_t off = 0, toff = 0;
    for (int e = 0; e < E; ++e) {
      r.offsets[e] = off;
      r.tile_off[e] = toff;
      r.counts[e] = cnt[e];
      cur[e] = off;
      off += cnt[e];
      toff += (cnt[e] + tile_tokens - 1) / tile_tokens;
    }
    r.offsets[E] = off;
    r.tile_off[E] = toff;
    r.flag[0] = bad;
  }
  __syncthreads();
  for (int64_t i = tid; i < npairs; i += blockDim.x) {
    const int e = ids[i];
    if (e >= 0 && e < E) {
      const int pos = atomicAdd(&cur[e], 1);
      r.perm[pos] = static_cast<int32_t>(i);
    }
  }
}

size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

// One warp per gathered row: 16-byte code chunks and the row's scales.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint8_t* __restrict__ codes,
                                                          const float* __restrict__ scales, int64_t K,
                                                          int top_k, int act_per_slot, Routing r, int E,
                                                          uint8_t* __restrict__ gcodes, float* __restrict__ gscales) {
  const int64_t rows = r.offsets[E];
  const int64_t B = K / 32;
  const int lane = threadIdx.x & 31;
  const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t i = w0; i < rows; i += nw) {
    const int64_t pr = r.perm[i];
    const int64_t src = act_per_slot ? pr : pr / top_k;
    const uint4* s = reinterpret_cast<const uint4*>(codes + src * (K / 2));
    uint4* d = reinterpret_cast<uint4*>(gcodes + i * (K / 2));
    for (int64_t c = lane; c < B; c += 32) d[c] = s[c];
    const float* ss = scales + src * B;
    float* ds = gscales + i * B;
    for (int64_t c = lane; c < B; c += 32) ds[c] = ss[c];
  }
}

}  // namespace

#ifndef W4A4_ROUTED_TILE_MULT
#define W4A4_ROUTED_TILE_MULT 2
#endif
int routed_tile_tokens(int64_t npairs, int E) {
  // about one tile per expert: twice the mean number of rows an expert receives,
  // in 32s, so that an expert a little above the mean still takes one tile (its
  // weights are converted once per weight tile, not twice)
  const int64_t mean = W4A4_ROUTED_TILE_MULT * ((npairs + E - 1) / E);
  int64_t t = (mean + 31) & ~int64_t(31);
  if (t < 32) t = 32;
  if (t > kRoutedTileMax) t = kRoutedTileMax;
  return static_cast<int>(t);
}

RoutingLayout routing_layout(int64_t npairs, int E, int64_t K) {
  RoutingLayout L{};
  size_t off = 0;
  L.flag = off;     off += 16;  // first, so that a status query needs only the pointer
  L.counts = off;   off += align16(sizeof(int32_t) * static_cast<size_t>(E));
  L.offsets = off;  off += align16(sizeof(int32_t) * static_cast<size_t>(E + 1));
  L.tile_off = off; off += align16(sizeof(int32_t) * static_cast<size_t>(E + 1));
  L.perm = off;     off += align16(sizeof(int32_t) * static_cast<size_t>(npairs));
  L.gcodes = off;   off += align16(static_cast<size_t>(npairs) * static_cast<size_t>(K / 2));
  L.gscales = off;  off += align16(static_cast<size_t>(npairs) * static_cast<size_t>(K / 32) * sizeof(float));
  L.total = off;
  return L;
}

Routing routing_in(void* ws, int64_t npairs, int E, int64_t K) {
  const RoutingLayout L = routing_layout(npairs, E, K);
  uint8_t* base = static_cast<uint8_t*>(ws);
  Routing r;
  r.counts = reinterpret_cast<int32_t*>(base + L.counts);
  r.offsets = reinterpret_cast<int32_t*>(base + L.offsets);
  r.tile_off = reinterpret_cast<int32_t*>(base + L.tile_off);
  r.perm = reinterpret_cast<int32_t*>(base + L.perm);
  r.flag = reinterpret_cast<int32_t*>(base + L.flag);
  r.gcodes = base + L.gcodes;
  r.gscales = reinterpret_cast<float*>(base + L.gscales);
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

cudaError_t launch_gemm_id(const uint8_t* w_codes, const uint16_t* w_scales, const int16_t* w_sums,
                           const uint8_t* w_expanded, int E, int64_t N, const uint8_t* a_codes, const float* a_scales,
                           int64_t K, const int32_t* ids, int64_t M, int top_k, int act_per_slot, float* y,
                           const Routing& r, cudaStream_t stream) {
  const int64_t npairs = M * top_k;
  const size_t sh = sizeof(int32_t) * 2 * static_cast<size_t>(E);
  const int tile = routed_tile_tokens(npairs, E);
  route_prep_kernel<<<1, kPrepThreads, sh, stream>>>(ids, npairs, E, N, tile, y, r);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t gwarps = npairs < 4096 * 8 ? npairs : 4096 * 8;
  gather_rows_kernel<<<static_cast<unsigned>((gwarps + 7) / 8), 256, 0, stream>>>(a_codes, a_scales, K, top_k,
                                                                                 act_per_slot, r, E, r.gcodes,
                                                                                 r.gscales);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_gemm_tc_routed(w_codes, w_scales, w_sums, w_expanded, E, N, r.gcodes, r.gscales, K, npairs, tile, y, r,
                               stream);
}

}  // namespace w4a4
