// Throughput probes for the roofline denominators the W4A4 path needs and the
// measured peaks do not carry: integer and fp8 warp-level MMA
// (mma.sync), fp8 tcgen05.mma, and the fp32 FMA pipe (scalar and f32x2).
// Built into a separate library (libw4a4_probes.so); not part of the W4A4 path.
//
// Each probe fills every SM, runs a long chain of independent operations and
// returns operations per second measured with CUDA events (0 on failure).
#include <cstdint>
#include <cstdio>
#include <cuda_runtime.h>

namespace {

constexpr int kChains = 8;

template <int KIND>
__global__ void mma_sync_probe(int iters, float* sink) {
  uint32_t a[4], b[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) a[i] = 0x01010101u * (threadIdx.x + i);
  b[0] = 0x02020202u;
  b[1] = 0x01010101u;
  float cf[kChains][4] = {};
  int ci[kChains][4] = {};
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int c = 0; c < kChains; ++c) {
      if constexpr (KIND == 0) {
        asm volatile("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
                     : "+r"(ci[c][0]), "+r"(ci[c][1]), "+r"(ci[c][2]), "+r"(ci[c][3])
                     : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
      } else if constexpr (KIND == 1) {
        asm volatile("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
                     : "+f"(cf[c][0]), "+f"(cf[c][1]), "+f"(cf[c][2]), "+f"(cf[c][3])
                     : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
      } else {
        asm volatile("mma.sync.aligned.m16n8k64.row.col.s32.s4.s4.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
                     : "+r"(ci[c][0]), "+r"(ci[c][1]), "+r"(ci[c][2]), "+r"(ci[c][3])
                     : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
      }
    }
  }
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < kChains; ++c)
#pragma unroll
    for (int j = 0; j < 4; ++j) s += cf[c][j] + static_cast<float>(ci[c][j]);
  if (s == 1.2345f) sink[threadIdx.x] = s;
}

template <bool PAIRED>
__global__ void ffma_probe(int iters, float* sink) {
  float x[kChains], y[kChains];
#pragma unroll
  for (int c = 0; c < kChains; ++c) {
    x[c] = threadIdx.x * 1e-7f + c;
    y[c] = c * 0.5f;
  }
  const float m = 0.9999f, ad = 1e-6f;
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int c = 0; c < kChains; c += 2) {
      if constexpr (PAIRED) {
        unsigned long long v, mm, aa;
        asm volatile("mov.b64 %0, {%1,%2};" : "=l"(v) : "f"(x[c]), "f"(x[c + 1]));
        asm volatile("mov.b64 %0, {%1,%2};" : "=l"(mm) : "f"(m), "f"(m));
        asm volatile("mov.b64 %0, {%1,%2};" : "=l"(aa) : "f"(ad), "f"(ad));
        asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(v) : "l"(mm), "l"(aa));
        asm volatile("mov.b64 {%0,%1}, %2;" : "=f"(x[c]), "=f"(x[c + 1]) : "l"(v));
        asm volatile("mov.b64 %0, {%1,%2};" : "=l"(v) : "f"(y[c]), "f"(y[c + 1]));
        asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(v) : "l"(mm), "l"(aa));
        asm volatile("mov.b64 {%0,%1}, %2;" : "=f"(y[c]), "=f"(y[c + 1]) : "l"(v));
      } else {
        asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(x[c]) : "f"(m), "f"(ad));
        asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(x[c + 1]) : "f"(m), "f"(ad));
        asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(y[c]) : "f"(m), "f"(ad));
        asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(y[c + 1]) : "f"(m), "f"(ad));
      }
    }
  }
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < kChains; ++c) s += x[c] + y[c];
  if (s == 1.2345f) sink[threadIdx.x] = s;
}

// ---- tcgen05 fp8 MMA: one CTA per SM, M=128 N=256 K=32 per instruction, zero operands.
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t desc_kmajor_noswizzle(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version for sm_100-family
  return d;                              // base offset 0, no swizzle
}

__global__ void __launch_bounds__(128) tcgen05_f8_probe(int iters, int* status) {
  __shared__ __align__(1024) uint8_t a_s[128 * 32];
  __shared__ __align__(1024) uint8_t b_s[256 * 32];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x;
  for (int i = tid; i < 128 * 32 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(a_s)[i] = 0u;
  for (int i = tid; i < 256 * 32 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(b_s)[i] = 0u;
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::);
  if (tid < 32) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(smem_u32(&tmem_base)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::);
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::);
  const uint32_t tmem = tmem_base;
  // instruction descriptor: D f32, A/B e4m3, K-major both, N = 256, M = 128
  const uint32_t idesc = (1u << 4) | (0u << 7) | (0u << 10) | ((256u >> 3) << 17) | ((128u >> 4) << 24);
  const uint64_t adesc = desc_kmajor_noswizzle(smem_u32(a_s), 128, 256);
  const uint64_t bdesc = desc_kmajor_noswizzle(smem_u32(b_s), 128, 256);
  if (tid == 0) {
    for (int it = 0; it < iters; ++it) {
      asm volatile(
          "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
          "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem),
          "l"(adesc), "l"(bdesc), "r"(idesc), "r"(it));
    }
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(&bar)));
  }
  // bounded wait for the MMAs (phase 0): at most one second of globaltimer
  uint32_t done = 0;
  uint64_t t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (uint64_t now = t0; !done && now - t0 < 1000000000ull;) {
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done) : "r"(smem_u32(&bar)), "r"(0u));
  }
  if (!done && tid == 0) atomicExch(status, 1);
  asm volatile("tcgen05.fence::before_thread_sync;" ::);
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::);
  if (tid < 32) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(tmem));
}


// Lane layout of the 16x256b TMEM load, read back from a known pattern.  One CTA
// of 4 warps allocates 32 columns; warp w writes its lane quarter with the
// 32x32b store (thread t <-> lane 32w + t, register j <-> column j), the value
// lane * 256 + column, then loads lanes 32w..32w+15 and 32w+16..32w+31 with
// 16x256b.x1 and records the 4 + 4 registers of every thread: out[128][8].
__global__ void __launch_bounds__(128) tmem_layout_probe(uint32_t* out) {
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 32;" ::"r"(smem_u32(&tmem_base)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::);
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::);
  const uint32_t tmem = tmem_base;
  const uint32_t row = static_cast<uint32_t>(32 * warp + lane);
  const uint32_t quarter = tmem + (static_cast<uint32_t>(32 * warp) << 16);
  uint32_t v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = row * 256u + static_cast<uint32_t>(j);
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(quarter), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]));
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
  uint32_t a[4], b[4];
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x1.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]) : "r"(quarter));
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x1.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]) : "r"(quarter + (16u << 16)));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    out[tid * 8 + j] = a[j];
    out[tid * 8 + 4 + j] = b[j];
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::);
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::);
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 32;" ::"r"(tmem));
}

template <typename F>
double time_kernel(F launch) {
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) return -1.0;
  launch();  // warm-up
  if (cudaDeviceSynchronize() != cudaSuccess) return -1.0;
  cudaEventRecord(e0);
  launch();
  cudaEventRecord(e1);
  if (cudaEventSynchronize(e1) != cudaSuccess) return -1.0;
  float ms = 0.f;
  cudaEventElapsedTime(&ms, e0, e1);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (cudaGetLastError() != cudaSuccess) return -1.0;
  return ms * 1e-3;
}

int sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n;
}

}  // namespace

extern "C" {

// kind: 0 = s8 m16n8k32, 1 = e4m3 m16n8k32, 2 = s4 m16n8k64.  Returns dense ops/s.
double w4a4_probe_mma_sync(int kind, int iters) {
  float* sink = nullptr;
  if (cudaMalloc(&sink, 4096) != cudaSuccess) return 0.0;
  const int blocks = sms() * 4, threads = 256;
  double s = time_kernel([&] {
    if (kind == 0) mma_sync_probe<0><<<blocks, threads>>>(iters, sink);
    else if (kind == 1) mma_sync_probe<1><<<blocks, threads>>>(iters, sink);
    else mma_sync_probe<2><<<blocks, threads>>>(iters, sink);
  });
  cudaFree(sink);
  if (s <= 0) return 0.0;
  const double k = (kind == 2) ? 64.0 : 32.0;
  const double ops = 2.0 * 16 * 8 * k * kChains * static_cast<double>(iters) * (blocks * threads / 32);
  return ops / s;
}

// paired: 0 = fma.rn.f32, 1 = fma.rn.f32x2.  Returns fp32 flop/s (2 per FMA lane).
double w4a4_probe_ffma(int paired, int iters) {
  float* sink = nullptr;
  if (cudaMalloc(&sink, 4096) != cudaSuccess) return 0.0;
  const int blocks = sms() * 8, threads = 256;
  double s = time_kernel([&] {
    if (paired) ffma_probe<true><<<blocks, threads>>>(iters, sink);
    else ffma_probe<false><<<blocks, threads>>>(iters, sink);
  });
  cudaFree(sink);
  if (s <= 0) return 0.0;
  const double flops = 2.0 * 2 * kChains * static_cast<double>(iters) * blocks * threads;
  return flops / s;
}

// Returns dense fp8 flop/s of tcgen05.mma kind::f8f6f4 (M128 N256 K32), or 0 on
// failure / timeout (status != 0).
double w4a4_probe_tcgen05_f8(int iters) {
  int* status = nullptr;
  if (cudaMalloc(&status, sizeof(int)) != cudaSuccess) return 0.0;
  cudaMemset(status, 0, sizeof(int));
  const int blocks = sms();
  double s = time_kernel([&] { tcgen05_f8_probe<<<blocks, 128>>>(iters, status); });
  int h = 1;
  cudaMemcpy(&h, status, sizeof(int), cudaMemcpyDeviceToHost);
  cudaFree(status);
  if (s <= 0 || h != 0) return 0.0;
  const double flops = 2.0 * 128 * 256 * 32 * static_cast<double>(iters) * blocks;
  return flops / s;
}


// The 16x256b TMEM load's register layout: out (host, 128 x 8 words) receives,
// per thread of 4 warps, the lane * 256 + column values of its 4 + 4 registers
// (lanes 32w.. and 32w + 16.. of its warp's quarter).  0 on success.
int w4a4_probe_tmem_layout(uint32_t* out) {
  uint32_t* d = nullptr;
  if (cudaMalloc(&d, 128 * 8 * sizeof(uint32_t)) != cudaSuccess) return 1;
  tmem_layout_probe<<<1, 128>>>(d);
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(out, d, 128 * 8 * sizeof(uint32_t), cudaMemcpyDeviceToHost);
  cudaFree(d);
  return e == cudaSuccess ? 0 : 2;
}

}  // extern "C"
