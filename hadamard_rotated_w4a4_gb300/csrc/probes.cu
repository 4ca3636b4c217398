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

#include "tc_ptx.cuh"

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


// Latency of one tcgen05.mma kind::f8f6f4 (M = 128, K = 32), issue to the
// completion its commit signals, in clock64 cycles: thread 0 issues it on zero
// operands (K-major, no swizzle, 8-row groups `sbo` bytes apart) and spins on the
// mbarrier.  Meanwhile warps 1-8 (`loaders` bit 0) stream 16x256b TMEM loads from
// the other 256 columns, as a fold would, and (bit 1) 16-byte shared-memory loads.
// out[rep] for 32 repetitions.
__global__ void __launch_bounds__(288) mma_latency_probe(int n, int sbo, int loaders, unsigned long long* out,
                                                         int* status, const uint8_t* gsrc, int64_t gbytes) {
  extern __shared__ __align__(1024) uint8_t dyn[];
  uint8_t* a_s = dyn;                // 16 groups x sbo bytes
  uint8_t* b_s = dyn + 16 * 1024;    // 32 groups x sbo bytes
  __shared__ __align__(8) uint64_t bar;
  __shared__ __align__(8) uint64_t cbar;
  __shared__ __align__(8) uint64_t bar2;
  __shared__ uint32_t tmem_base;
  __shared__ volatile int stop;
  __shared__ volatile int ack;
  __shared__ volatile unsigned long long t_obs;
  uint8_t* c_s = dyn + 48 * 1024;  // bulk-copy destination, 48 KB
  const int tid = threadIdx.x, warp = tid >> 5;
  // operands: zero (fill 0) or a pattern of nonzero e4m3 values (fill 1: bytes 0x01..0x0F and 0x81..0x8F)
  for (int i = tid; i < (16 + 32) * 1024 / 4; i += blockDim.x) {
    const uint32_t h = static_cast<uint32_t>(i) * 2654435761u;
    reinterpret_cast<uint32_t*>(dyn)[i] = (loaders & 4) ? ((h & 0x0F0F0F0Fu) | 0x01010101u) | (h & 0x80808080u) : 0u;
  }
  if (tid == 0) {
    stop = 0;
    ack = 0;
    t_obs = 0;
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar)));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&cbar)));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar2)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::);
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&tmem_base)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::);
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::);
  const uint32_t tmem = tmem_base;
  const uint32_t idesc = (1u << 4) | ((static_cast<uint32_t>(n) >> 3) << 17) | ((128u >> 4) << 24);
  const uint64_t adesc = desc_kmajor_noswizzle(smem_u32(a_s), 128, sbo);
  const uint64_t bdesc = desc_kmajor_noswizzle(smem_u32(b_s), 128, sbo);
  if (warp == 0) {
    if (tid == 0) {
      int bad = 0;
      for (int rep = 0; rep < 32; ++rep) {
        unsigned long long t0, t1;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("mov.u64 %0, %%clock64;" : "=l"(t0));
        asm volatile(
            "{\n.reg .pred p;\nsetp.ne.b32 p, 0, 0;\n"
            "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc));
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(&bar)));
        uint32_t done = 0;
        const uint32_t parity = rep & 1;
        if (loaders & 16) {  // warp 1 observes the completion; this thread waits for its word
          if (loaders & 32) {  // first 3000 cycles of plain busy work
            unsigned long long tb;
            do {
              asm volatile("mov.u64 %0, %%clock64;" : "=l"(tb));
            } while (tb - t0 < 3000);
          }
          if (loaders & 64) {  // wait on a second barrier that the observer arrives on
            for (long spin = 0; !done && spin < 100000000L; ++spin) {
              if (loaders & 128)
                asm volatile(
                    "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, "
                    "p;\n}\n"
                    : "=r"(done) : "r"(smem_u32(&bar2)), "r"(parity) : "memory");
              else
                asm volatile(
                    "{\n.reg .pred p;\nmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, "
                    "p;\n}\n"
                    : "=r"(done) : "r"(smem_u32(&bar2)), "r"(parity) : "memory");
            }
          } else {
            for (long spin = 0; !done && spin < 100000000L; ++spin) done = ack == rep + 1;
          }
          t1 = t_obs;
        } else {
          for (long spin = 0; !done && spin < 100000000L; ++spin) {
            asm volatile(
                "{\n.reg .pred p;\nmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                : "=r"(done) : "r"(smem_u32(&bar)), "r"(parity));
          }
          asm volatile("mov.u64 %0, %%clock64;" : "=l"(t1));
        }
        if (!done) bad = 1;
        out[rep] = t1 - t0;
        if (bad) break;
      }
      if (bad) atomicExch(status, 1);
      stop = 1;
    }
    __syncwarp();
  } else if ((loaders & 16) && warp == 1) {  // the completion observer
    if ((tid & 31) == 0) {
      for (int rep = 0; rep < 32 && !stop; ++rep) {
        uint32_t done = 0;
        for (long spin = 0; !done && spin < 100000000L; ++spin)
          asm volatile(
              "{\n.reg .pred p;\nmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
              : "=r"(done) : "r"(smem_u32(&bar)), "r"(static_cast<uint32_t>(rep & 1)));
        unsigned long long t;
        asm volatile("mov.u64 %0, %%clock64;" : "=l"(t));
        t_obs = t;
        __threadfence_block();
        if (loaders & 64)
          asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&bar2)) : "memory");
        else
          ack = rep + 1;
        if (!done) break;
      }
    }
    __syncwarp();
  } else if ((loaders & 8) && warp == 8) {  // warp 8: 48 KB bulk copies from global memory, back to back
    if ((tid & 31) == 0) {
      int64_t off = 0;
      for (long it = 0; !stop && it < 1000000L; ++it) {
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(&cbar)), "r"(48 * 1024)
                     : "memory");
        for (int c = 0; c < 3; ++c)
          asm volatile(
              "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                  smem_u32(c_s + c * 16384)),
              "l"(gsrc + off + c * 16384), "r"(16384), "r"(smem_u32(&cbar))
              : "memory");
        off = (off + 48 * 1024) % (gbytes - 48 * 1024);
        uint32_t done = 0;
        for (long spin = 0; !done && spin < 100000000L; ++spin)
          asm volatile(
              "{\n.reg .pred p;\nmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
              : "=r"(done) : "r"(smem_u32(&cbar)), "r"(static_cast<uint32_t>(it & 1)));
      }
    }
    __syncwarp();
  } else if (loaders & 3) {  // warps 1-8: TMEM loads from columns 256.. of their lane quarter, and/or shared loads
    const uint32_t quarter = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + 256u;
    uint32_t acc = 0;
    for (long it = 0; !stop && it < 100000000L; ++it) {
      if (loaders & 1) {
        uint32_t r[16];
        const uint32_t col = static_cast<uint32_t>((it & 7) * 32);
        asm volatile(
            "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
            : "r"(quarter + col));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        for (int j = 0; j < 16; ++j) acc += r[j];
      }
      if (loaders & 2) {
        uint32_t v0, v1, v2, v3;
        asm volatile("ld.volatile.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3)
                     : "r"(smem_u32(dyn + ((tid * 16 + it * 512) & (48 * 1024 - 1)))));
        acc += v0 + v3;
      }
    }
    if (acc == 12345u) out[40] = acc;
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::);
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::);
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
}


// Issue rate of back-to-back fp8 MMAs from one thread: `iters` MMAs of M 128, N n,
// K 32, a commit after every `per_commit` of them; the clock after each issue.
// flags bit 0: alternate two 256-column TMEM buffers; bit 1: warps 1-8 run a
// fused multiply-add loop meanwhile (paired fp32, as the fold does); bit 2:
// accumulate into D (from the third MMA on); bit 3: no clock reads between issues;
// bit 4: zero operands; bit 5: every operand byte 0x01; bit 6: one CTA per SM
// (block 0 timed); bit 7: 256 TMEM columns (the two buffers 128 apart); bit 8:
// 128-byte swizzled operands; bit 9: unswizzled, 8-row groups 1024 bytes apart.
__global__ void __launch_bounds__(288) mma_rate_probe(int n, int per_commit, int iters, int flags,
                                                      unsigned long long* out, int* status) {
  extern __shared__ __align__(1024) uint8_t dyn[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_base;
  __shared__ volatile int stop;
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int i = tid; i < 48 * 1024 / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(dyn)[i] = (flags & 16) ? 0u : (flags & 32) ? 0x01010101u : 0x01020304u;
  if (tid == 0) {
    stop = 0;
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::);
  if (warp == 0) {
    if (flags & 128)
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(smem_u32(&tmem_base)));
    else
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&tmem_base)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::);
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::);
  const uint32_t tmem = tmem_base;
  const uint32_t idesc = (1u << 4) | ((static_cast<uint32_t>(n) >> 3) << 17) | ((128u >> 4) << 24);
  // operands: bit 8, the 128-byte swizzle (A 16 KB at 0, B 32 KB at 16 KB, 128-byte
  // rows), K step k at byte 32k of the row; bit 9, no swizzle with 8-row groups 1024
  // bytes apart; else no swizzle, groups 256 bytes apart
  const uint64_t adesc = (flags & 256) ? w4a4::kmajor_desc_sw128(dyn)
                         : (flags & 512) ? desc_kmajor_noswizzle(smem_u32(dyn), 128, 1024)
                                         : desc_kmajor_noswizzle(smem_u32(dyn), 128, 256);
  const uint64_t bdesc = (flags & 256) ? w4a4::kmajor_desc_sw128(dyn + 16384)
                         : (flags & 512) ? desc_kmajor_noswizzle(smem_u32(dyn + 16384), 128, 1024)
                                         : desc_kmajor_noswizzle(smem_u32(dyn + 16384), 128, 256);
  if (warp == 0) {
    if (tid == 0) {
      unsigned long long t;
      int commits = 0;
      asm volatile("mov.u64 %0, %%clock64;" : "=l"(t));
      if (blockIdx.x == 0) out[0] = t;
      int cnt = 0;
      const uint32_t alt = (flags & 1) ? 128u : 0u;
      const int acc_from = (flags & 4) ? 2 : iters;
      for (int i = 0; i < iters; ++i) {
        const uint32_t d = tmem + ((i & 1) ? alt : 0u);
        const uint32_t acc = static_cast<uint32_t>(i >= acc_from);
        const uint64_t koff = (flags & 768) ? static_cast<uint64_t>(2 * (i & 3)) : 0u;  // 32 bytes >> 4
        asm volatile(
            "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
            "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
            "l"(adesc + koff), "l"(bdesc + koff), "r"(idesc), "r"(acc));
        if (++cnt == per_commit || i + 1 == iters) {
          cnt = 0;
          asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
              smem_u32(&bar)));
          ++commits;
        }
        if (!(flags & 8)) {
          asm volatile("mov.u64 %0, %%clock64;" : "=l"(t));
          if (i < 60 && blockIdx.x == 0) out[1 + i] = t;
        }
      }
      // every commit's phase: wait for the last one (count 1: one phase per commit)
      uint32_t done = 0;
      for (long spin = 0; !done && spin < 100000000L; ++spin)
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done) : "r"(smem_u32(&bar)), "r"(static_cast<uint32_t>((commits - 1) & 1)));
      asm volatile("mov.u64 %0, %%clock64;" : "=l"(t));
      if (blockIdx.x == 0) out[61] = t;
      if (!done) atomicExch(status, 1);
      stop = 1;
    }
    __syncwarp();
  } else if (flags & 2) {
    float2 a = make_float2(tid, 1.f), b = make_float2(0.5f, 0.25f), c0 = make_float2(0.f, 0.f), c1 = c0, c2 = c0,
           c3 = c0;
    for (long it = 0; !stop && it < 10000000L; ++it) {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        c0 = __ffma2_rn(a, b, c0);
        c1 = __ffma2_rn(a, c0, c1);
        c2 = __ffma2_rn(b, c1, c2);
        c3 = __ffma2_rn(a, c2, c3);
      }
    }
    if (c3.x == 12345.f) out[62] = 1;
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::);
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::);
  if (warp == 0) {
    if (flags & 128)
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(tmem));
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
  }
}


// TMEM load latency: warps 0..nwarps-1 each time `reps` back-to-back
// (tcgen05.ld + tcgen05.wait::ld) of the 16x256b shape, .x4 (x8 = 0) or .x8
// (x8 = 1), from their lane quarter of a 512-column allocation.
__global__ void __launch_bounds__(256) tmem_ld_probe(int x8, int nwarps, int reps, unsigned long long* out) {
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&tmem_base)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::);
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::);
  const uint32_t tmem = tmem_base + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
  uint32_t acc = 0;
  if (warp < nwarps) {
    unsigned long long t0, t1;
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(t0));
    for (int it = 0; it < reps; ++it) {
      const uint32_t col = static_cast<uint32_t>((it & 3) * 128);
      if (x8) {
        uint32_t r[32];
        w4a4::tmem_ld16x256_x8(tmem + col, r);
        w4a4::tmem_wait32(r);
#pragma unroll
        for (int j = 0; j < 32; ++j) acc += r[j];
      } else {
        uint32_t r[16];
        w4a4::tmem_ld16x256_x4(tmem + col, r);
        w4a4::tmem_wait(r);
#pragma unroll
        for (int j = 0; j < 16; ++j) acc += r[j];
      }
    }
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(t1));
    if ((tid & 31) == 0) out[warp] = t1 - t0;
  }
  if (acc == 0x12345678u) out[63] = acc;
  asm volatile("tcgen05.fence::before_thread_sync;" ::);
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::);
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem_base));
}


// The bare MMA -> fold handshake: warp 0 lane 0 issues one M 128, N 256, K 32
// fp8 MMA per block into TMEM buffer b % 2 (after the buffer's release) and
// commits it; warps 1-8 wait for each block and hand its buffer back.  flags bit
// 0: the consumers wait with try_wait (else test_wait polls); bit 1: each
// consumer warp loads one 16x256b.x4 piece of the block first; bit 2: the
// issuer waits with try_wait.  out[0] = cycles per block seen by warp 1.
__global__ void __launch_bounds__(288) pipe_probe(int nblocks, int flags, unsigned long long* out, int* status) {
  extern __shared__ __align__(1024) uint8_t dyn[];
  __shared__ __align__(8) uint64_t full[2], empty[2];
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < 48 * 1024 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(dyn)[i] = 0x01020304u;
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&full[i])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 8;" ::"r"(smem_u32(&empty[i])));
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::);
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&tmem_base)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::);
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::);
  const uint32_t tmem = tmem_base;
  const uint32_t idesc = (1u << 4) | ((256u >> 3) << 17) | ((128u >> 4) << 24);
  const uint64_t adesc = desc_kmajor_noswizzle(smem_u32(dyn), 128, 256);
  const uint64_t bdesc = desc_kmajor_noswizzle(smem_u32(dyn + 16384), 128, 256);
  const long kSpin = 20000000L;
  if (warp == 0) {
    if (lane == 0) {
      for (int b = 0; b < nblocks; ++b) {
        const int tb = b & 1;
        uint32_t ok = 0;
        const uint32_t par = ((b >> 1) & 1) ^ 1;
        for (long n = 0; !ok && n < kSpin; ++n) {
          if (flags & 4)
            asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                         : "=r"(ok) : "r"(smem_u32(&empty[tb])), "r"(par) : "memory");
          else
            asm volatile("{\n.reg .pred p;\nmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                         : "=r"(ok) : "r"(smem_u32(&empty[tb])), "r"(par) : "memory");
        }
        if (!ok) { atomicExch(status, 1); break; }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, 0, 0;\ntcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n"
                     ::"r"(tmem + static_cast<uint32_t>(tb * 256)), "l"(adesc), "l"(bdesc), "r"(idesc));
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(&full[tb])) : "memory");
      }
    }
    __syncwarp();
  } else if (warp <= 8) {
    unsigned long long t0 = 0, t1;
    uint32_t acc = 0;
    const uint32_t q = static_cast<uint32_t>(warp & 3);
    for (int b = 0; b < nblocks; ++b) {
      const int tb = b & 1;
      uint32_t ok = 0;
      const uint32_t par = (b >> 1) & 1;
      for (long n = 0; !ok && n < kSpin; ++n) {
        if (flags & 1)
          asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                       : "=r"(ok) : "r"(smem_u32(&full[tb])), "r"(par) : "memory");
        else
          asm volatile("{\n.reg .pred p;\nmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                       : "=r"(ok) : "r"(smem_u32(&full[tb])), "r"(par) : "memory");
      }
      if (!ok) { atomicExch(status, 2); break; }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      if (b == 16 && warp == 1 && lane == 0) asm volatile("mov.u64 %0, %%clock64;" : "=l"(t0));
      if (flags & 2) {
        uint32_t r[16];
        w4a4::tmem_ld16x256_x4(tmem + (q << 21) + static_cast<uint32_t>(tb * 256 + 32 * (warp >> 2)), r);
        w4a4::tmem_wait(r);
        acc += r[0] ^ r[15];
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&empty[tb])) : "memory");
    }
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(t1));
    if (warp == 1 && lane == 0 && nblocks > 16) out[0] = (t1 - t0) / static_cast<unsigned long long>(nblocks - 16);
    if (acc == 0x12345u) out[1] = acc;
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::);
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::);
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
}


// The fold alone: warps fold `nblocks` 128 x 256 accumulator blocks read from
// TMEM (two 256-column buffers, alternating) with the GEMM's per-piece loop --
// 16x256b.x4 loads one piece ahead, paired FMAs t = fma(D, dw, c), acc = fma(t,
// da, acc) with scales from shared memory -- and no barrier.  out[w] = cycles per
// block of warp w.
template <int NW, int mode>
__global__ void __launch_bounds__(32 * NW) fold_probe(int nblocks, unsigned long long* out) {
  // mode bit 0: no TMEM loads (registers from the loop index); bit 1: scales from
  // registers (no shared loads); bit 2: 16 warps, each with half the columns
  // (chunks hq and hq + 4 of the 8), else 8 warps with four chunks each.
  __shared__ uint32_t tmem_base;
  __shared__ __align__(16) float sc[4096];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int nw = NW;
  constexpr int NKK = NW == 16 ? 2 : 4;  // chunks per warp
  for (int i = tid; i < 4096; i += blockDim.x) sc[i] = 1.0f + 0.001f * (i & 63);
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&tmem_base)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::);
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::);
  const int q = warp & 3, h = warp >> 2, jr = lane >> 2, u = lane & 3;
  float2 acc[NKK][2][4][2];
#pragma unroll
  for (int a = 0; a < NKK; ++a)
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        acc[a][b][x][0] = make_float2(0.f, 0.f);
        acc[a][b][x][1] = make_float2(0.f, 0.f);
      }
  unsigned long long t0, t1;
  asm volatile("mov.u64 %0, %%clock64;" : "=l"(t0));
  {
    for (int bk = 0; bk < nblocks; ++bk) {
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>((bk & 1) * 256);
      const float* sb = sc + (bk & 7) * 512;
      float4 dwv, crv;
      if constexpr ((mode & 2) != 0) {
        dwv = make_float4(1.f + bk, 2.f, 3.f, 4.f);
        crv = make_float4(0.5f, 0.25f + bk, 0.125f, 1.f);
      } else {
        dwv = *reinterpret_cast<const float4*>(sb + 32 * q + 4 * jr);
        crv = *reinterpret_cast<const float4*>(sb + 128 + 32 * q + 4 * jr);
      }
      uint32_t ra[16], rb[16];
      constexpr int np = 2 * NKK;
      if constexpr ((mode & 1) == 0) {
        w4a4::tmem_ld16x256_x4(tbase + static_cast<uint32_t>(32 * h), ra);
        w4a4::tmem_wait(ra);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) ra[i] = __float_as_uint(1.0f + i + bk);
      }
      float4 da0 = make_float4(0.f, 0.f, 0.f, 0.f), da1 = da0;
#pragma unroll
      for (int pc = 0; pc < np; ++pc) {
        const int kk = pc >> 1, hf = pc & 1;
        const int kcol = NW == 16 ? h + 4 * kk : h + 2 * kk;
        uint32_t(&cur)[16] = (pc & 1) ? rb : ra;
        uint32_t(&nxt)[16] = (pc & 1) ? ra : rb;
        if (pc + 1 < np) {
          const int k1 = NW == 16 ? h + 4 * ((pc + 1) >> 1) : h + 2 * ((pc + 1) >> 1), hf1 = (pc + 1) & 1;
          if constexpr ((mode & 1) == 0) {
            w4a4::tmem_ld16x256_x4(tbase + (static_cast<uint32_t>(16 * hf1) << 16) + static_cast<uint32_t>(32 * k1),
                                   nxt);
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) nxt[i] = __float_as_uint(2.0f + i + pc + bk);
          }
        }
        if (hf == 0) {
          if constexpr ((mode & 2) != 0) {
            da0 = make_float4(0.1f * kk, 0.2f, 0.3f, 0.4f + bk);
            da1 = make_float4(0.5f, 0.6f + bk, 0.7f, 0.8f);
          } else {
            const float4* dap = reinterpret_cast<const float4*>(sb + 256 + (32 * kcol) % 256 + 8 * u);
            da0 = dap[0];
            da1 = dap[1];
          }
        }
        const float dA = hf ? dwv.z : dwv.x, dB = hf ? dwv.w : dwv.y;
        const float cA = hf ? crv.z : crv.x, cB = hf ? crv.w : crv.y;
        const float2 dw0 = make_float2(dA, dA), dw1 = make_float2(dB, dB);
        const float2 c0 = make_float2(cA, cA), c1 = make_float2(cB, cB);
        const float2 dav[4] = {make_float2(da0.x, da0.y), make_float2(da0.z, da0.w), make_float2(da1.x, da1.y),
                               make_float2(da1.z, da1.w)};
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const float2 a0 =
              __ffma2_rn(make_float2(__uint_as_float(cur[4 * x]), __uint_as_float(cur[4 * x + 1])), dw0, c0);
          const float2 a1 =
              __ffma2_rn(make_float2(__uint_as_float(cur[4 * x + 2]), __uint_as_float(cur[4 * x + 3])), dw1, c1);
          acc[kk][hf][x][0] = __ffma2_rn(a0, dav[x], acc[kk][hf][x][0]);
          acc[kk][hf][x][1] = __ffma2_rn(a1, dav[x], acc[kk][hf][x][1]);
        }
        if constexpr ((mode & 1) == 0) {
          if (pc + 1 < np) w4a4::tmem_wait(nxt);
        }
      }
    }
  }
  asm volatile("mov.u64 %0, %%clock64;" : "=l"(t1));
  float sum = 0.f;
#pragma unroll
  for (int a = 0; a < NKK; ++a)
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
      for (int x = 0; x < 4; ++x) sum += acc[a][b][x][0].x + acc[a][b][x][1].y;
  if (lane == 0) out[warp] = (t1 - t0) / static_cast<unsigned long long>(nblocks);
  if (sum == 1234.5f) out[63] = 1;
  asm volatile("tcgen05.fence::before_thread_sync;" ::);
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::);
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem_base));
}


// The fold loop (8 warps, warps 4-11, as fold_probe mode 0 on TMEM columns
// 256..511) with warp 1 issuing `mma_per` back-to-back M 128 N 256 K 32 fp8 MMAs
// into columns 0..255 for every block the fold warps do (mma_per = 0: idle) and
// warp 0 issuing `tma_per` 4 KB bulk copies per block (0: idle).  out[w] = fold
// cycles per block of warp w (4..11), so the warps beside the issuers (SM
// sub-partitions 0 and 1) can be compared with the others.
__global__ void __launch_bounds__(384) fold_mma_probe(int nblocks, int mma_per, int tma_per, const uint8_t* gsrc,
                                                      unsigned long long* out, int* status) {
  extern __shared__ __align__(1024) uint8_t dyn[];
  __shared__ uint32_t tmem_base;
  __shared__ __align__(16) float sc[4096];
  __shared__ __align__(8) uint64_t mbar, cbar;
  __shared__ volatile int stop;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < 4096; i += blockDim.x) sc[i] = 1.0f + 0.001f * (i & 63);
  for (int i = tid; i < 48 * 1024 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(dyn)[i] = 0x01020304u;
  if (tid == 0) {
    stop = 0;
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&mbar)));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&cbar)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::);
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&tmem_base)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::);
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::);
  const uint32_t tmem = tmem_base;
  if (warp == 1) {
    if (lane == 0 && mma_per > 0) {
      const uint32_t idesc = (1u << 4) | ((256u >> 3) << 17) | ((128u >> 4) << 24);
      const uint64_t adesc = desc_kmajor_noswizzle(smem_u32(dyn), 128, 256);
      const uint64_t bdesc = desc_kmajor_noswizzle(smem_u32(dyn + 16384), 128, 256);
      uint32_t ph = 0;
      for (long it = 0; !stop && it < 4000000L; ++it) {
        for (int k = 0; k < mma_per; ++k)
          asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, 0, 0;\ntcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n"
                       ::"r"(tmem), "l"(adesc), "l"(bdesc), "r"(idesc));
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(&mbar)) : "memory");
        uint32_t done = 0;
        for (long n = 0; !done && n < 20000000L; ++n)
          asm volatile("{\n.reg .pred p;\nmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                       : "=r"(done) : "r"(smem_u32(&mbar)), "r"(ph) : "memory");
        if (!done) { atomicExch(status, 1); break; }
        ph ^= 1;
        // pace: about one group of MMAs per 700 cycles (a fold block)
        unsigned long long t0, t1;
        asm volatile("mov.u64 %0, %%clock64;" : "=l"(t0));
        do { asm volatile("mov.u64 %0, %%clock64;" : "=l"(t1)); } while (t1 - t0 < 500 && !stop);
      }
    }
    __syncwarp();
  } else if (warp == 0) {
    if (lane == 0 && tma_per > 0) {
      uint32_t ph = 0;
      for (long it = 0; !stop && it < 4000000L; ++it) {
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(&cbar)), "r"(4096 * tma_per) : "memory");
        for (int k = 0; k < tma_per; ++k)
          asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], 4096, [%2];"
                       ::"r"(smem_u32(dyn + 32768 + 4096 * (k & 3))), "l"(gsrc + (static_cast<int64_t>(it * tma_per + k) % 4096) * 4096),
                         "r"(smem_u32(&cbar)) : "memory");
        uint32_t done = 0;
        for (long n = 0; !done && n < 20000000L; ++n)
          asm volatile("{\n.reg .pred p;\nmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                       : "=r"(done) : "r"(smem_u32(&cbar)), "r"(ph) : "memory");
        if (!done) { atomicExch(status, 2); break; }
        ph ^= 1;
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    const int q = warp & 3, h = (warp - 4) >> 2, jr = lane >> 2, u = lane & 3;
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
    unsigned long long t0, t1;
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(t0));
    for (int bk = 0; bk < nblocks; ++bk) {
      const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * q) << 16) + 256u;
      const float* sb = sc + (bk & 7) * 512;
      const float4 dwv = *reinterpret_cast<const float4*>(sb + 32 * q + 4 * jr);
      const float4 crv = *reinterpret_cast<const float4*>(sb + 128 + 32 * q + 4 * jr);
      uint32_t ra[16], rb[16];
      w4a4::tmem_ld16x256_x4(tbase + static_cast<uint32_t>(32 * h), ra);
      w4a4::tmem_wait(ra);
      float4 da0, da1;
#pragma unroll
      for (int pc = 0; pc < 8; ++pc) {
        const int kk = pc >> 1, hf = pc & 1;
        uint32_t(&cur)[16] = (pc & 1) ? rb : ra;
        uint32_t(&nxt)[16] = (pc & 1) ? ra : rb;
        if (pc + 1 < 8) {
          const int k1 = h + 2 * ((pc + 1) >> 1), hf1 = (pc + 1) & 1;
          w4a4::tmem_ld16x256_x4(tbase + (static_cast<uint32_t>(16 * hf1) << 16) + static_cast<uint32_t>(32 * k1), nxt);
        }
        if (hf == 0) {
          const float4* dap = reinterpret_cast<const float4*>(sb + 256 + (32 * (h + 2 * kk)) % 256 + 8 * u);
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
          const float2 a0 = __ffma2_rn(make_float2(__uint_as_float(cur[4 * x]), __uint_as_float(cur[4 * x + 1])), dw0, c0);
          const float2 a1 =
              __ffma2_rn(make_float2(__uint_as_float(cur[4 * x + 2]), __uint_as_float(cur[4 * x + 3])), dw1, c1);
          acc[kk][hf][x][0] = __ffma2_rn(a0, dav[x], acc[kk][hf][x][0]);
          acc[kk][hf][x][1] = __ffma2_rn(a1, dav[x], acc[kk][hf][x][1]);
        }
        if (pc + 1 < 8) w4a4::tmem_wait(nxt);
      }
    }
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(t1));
    float sum = 0.f;
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int x = 0; x < 4; ++x) sum += acc[a][b][x][0].x + acc[a][b][x][1].y;
    if (lane == 0) out[warp] = (t1 - t0) / static_cast<unsigned long long>(nblocks);
    if (sum == 1234.5f) out[63] = 1;
  }
  // warps 4-11 meet at a named barrier (256 threads) once their fold is done; one of
  // them then tells the issuers to stop.  Warps 0-3 skip it.
  if (warp >= 4) {
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (tid == 128) stop = 1;
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::);
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::);
  if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
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


// One tcgen05 MMA's latency (clock64 cycles, median of 32 repetitions after 4) for
// M = 128, N = n, K = 32 fp8, K-major operands with 8-row groups sbo bytes apart;
// loaders: bit 0, eight other warps stream TMEM loads meanwhile; bit 1, shared-memory
// loads; bit 2, nonzero operands; bit 3, a warp streaming 48 KB bulk copies from
// global memory into shared memory; bit 4, the completion observed by another
// warp (the issuing thread waits for that warp's word); bit 5, with bit 4, the
// issuing thread busy for 3000 cycles first; bit 6, with bit 4, the issuing
// thread waits on a second mbarrier that the observer arrives on (test_wait
// polls; bit 7: try_wait).  -1 on failure.
double w4a4_probe_mma_latency(int n, int sbo, int loaders) {
  if (n < 16 || n > 256 || n % 16 || (sbo != 256 && sbo != 1024) || loaders < 0 || loaders > 255) return -1.0;
  unsigned long long* d = nullptr;
  int* status = nullptr;
  if (cudaMalloc(&d, 64 * sizeof(unsigned long long)) != cudaSuccess) return -1.0;
  if (cudaMalloc(&status, sizeof(int)) != cudaSuccess) { cudaFree(d); return -1.0; }
  cudaMemset(status, 0, sizeof(int));
  const size_t smem = (16 + 32 + 48) * 1024;
  const int64_t gbytes = int64_t(64) << 20;
  uint8_t* gsrc = nullptr;
  if (cudaMalloc(&gsrc, gbytes) != cudaSuccess) { cudaFree(d); cudaFree(status); return -1.0; }
  cudaMemset(gsrc, 0x11, gbytes);
  cudaFuncSetAttribute(mma_latency_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  mma_latency_probe<<<1, 288, smem>>>(n, sbo, loaders, d, status, gsrc, gbytes);
  unsigned long long h[64] = {};
  int hs = 1;
  const cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) {
    cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost);
    cudaMemcpy(&hs, status, sizeof(int), cudaMemcpyDeviceToHost);
  }
  cudaFree(d);
  cudaFree(status);
  cudaFree(gsrc);
  if (e != cudaSuccess || hs != 0) return -1.0;
  unsigned long long v[28];
  for (int i = 0; i < 28; ++i) v[i] = h[4 + i];
  for (int i = 1; i < 28; ++i)
    for (int j = i; j > 0 && v[j - 1] > v[j]; --j) {
      const unsigned long long t = v[j];
      v[j] = v[j - 1];
      v[j - 1] = t;
    }
  return static_cast<double>(v[14]);
}


// Back-to-back MMA issue (mma_rate_probe): out2[0] = median cycles between issues
// 10..59, out2[1] = cycles from the first issue to the last commit's completion
// divided by iters.  0 on success.
int w4a4_probe_mma_rate(int n, int per_commit, int iters, int flags, double* out2) {
  if (n < 16 || n > 256 || n % 16 || per_commit < 1 || iters < 61 || iters > 100000 || flags < 0 || flags > 1023 || (flags & 768) == 768)
    return -1;
  if ((flags & 1) && n > ((flags & 128) ? 128 : 256)) return -1;  // the second buffer must fit
  unsigned long long* d = nullptr;
  int* status = nullptr;
  if (cudaMalloc(&d, 64 * sizeof(unsigned long long)) != cudaSuccess) return -1;
  if (cudaMalloc(&status, sizeof(int)) != cudaSuccess) { cudaFree(d); return -1; }
  cudaMemset(d, 0, 64 * sizeof(unsigned long long));
  cudaMemset(status, 0, sizeof(int));
  const size_t smem = 48 * 1024;
  cudaFuncSetAttribute(mma_rate_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  mma_rate_probe<<<(flags & 64) ? sms() : 1, 288, smem>>>(n, per_commit, iters, flags, d, status);
  unsigned long long h[64] = {};
  int hs = 1;
  const cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) {
    cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost);
    cudaMemcpy(&hs, status, sizeof(int), cudaMemcpyDeviceToHost);
  }
  cudaFree(d);
  cudaFree(status);
  if (e != cudaSuccess || hs != 0) return -1;
  unsigned long long v[49];
  for (int i = 0; i < 49; ++i) v[i] = h[12 + i] - h[11 + i];
  for (int i = 1; i < 49; ++i)
    for (int j = i; j > 0 && v[j - 1] > v[j]; --j) {
      const unsigned long long t = v[j];
      v[j] = v[j - 1];
      v[j - 1] = t;
    }
  out2[0] = static_cast<double>(v[24]);
  out2[1] = static_cast<double>(h[61] - h[0]) / iters;
  return 0;
}


// Cycles per TMEM load + wait (tmem_ld_probe), averaged over the timed warps.
double w4a4_probe_tmem_ld(int x8, int nwarps, int reps) {
  if (nwarps < 1 || nwarps > 8 || reps < 1 || reps > 100000 || (x8 != 0 && x8 != 1)) return -1.0;
  unsigned long long* d = nullptr;
  if (cudaMalloc(&d, 64 * sizeof(unsigned long long)) != cudaSuccess) return -1.0;
  cudaMemset(d, 0, 64 * sizeof(unsigned long long));
  tmem_ld_probe<<<1, 256>>>(x8, nwarps, reps, d);
  unsigned long long h[64] = {};
  const cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost);
  cudaFree(d);
  if (e != cudaSuccess) return -1.0;
  double sum = 0;
  for (int w = 0; w < nwarps; ++w) sum += static_cast<double>(h[w]);
  return sum / nwarps / reps;
}


// Cycles per block of the bare MMA -> fold handshake (pipe_probe), -1 on failure.
double w4a4_probe_pipe(int nblocks, int flags) {
  if (nblocks < 32 || nblocks > 100000 || flags < 0 || flags > 7) return -1.0;
  unsigned long long* d = nullptr;
  int* status = nullptr;
  if (cudaMalloc(&d, 4 * sizeof(unsigned long long)) != cudaSuccess) return -1.0;
  if (cudaMalloc(&status, sizeof(int)) != cudaSuccess) { cudaFree(d); return -1.0; }
  cudaMemset(d, 0, 4 * sizeof(unsigned long long));
  cudaMemset(status, 0, sizeof(int));
  const size_t smem = 48 * 1024;
  cudaFuncSetAttribute(pipe_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  pipe_probe<<<1, 288, smem>>>(nblocks, flags, d, status);
  unsigned long long h[4] = {};
  int hs = 1;
  const cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) {
    cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost);
    cudaMemcpy(&hs, status, sizeof(int), cudaMemcpyDeviceToHost);
  }
  cudaFree(d);
  cudaFree(status);
  if (e != cudaSuccess || hs != 0) return -1.0;
  return static_cast<double>(h[0]);
}


// Cycles per 128 x 256 block of the fold alone (fold_probe, see its modes), mean
// over the warps.
double w4a4_probe_fold(int nblocks, int mode) {
  if (nblocks < 1 || nblocks > 100000 || mode < 0 || mode > 7) return -1.0;
  unsigned long long* d = nullptr;
  if (cudaMalloc(&d, 64 * sizeof(unsigned long long)) != cudaSuccess) return -1.0;
  cudaMemset(d, 0, 64 * sizeof(unsigned long long));
  const int nw = (mode & 4) ? 16 : 8;
  switch (mode) {
    case 0: fold_probe<8, 0><<<1, 256>>>(nblocks, d); break;
    case 1: fold_probe<8, 1><<<1, 256>>>(nblocks, d); break;
    case 2: fold_probe<8, 2><<<1, 256>>>(nblocks, d); break;
    case 3: fold_probe<8, 3><<<1, 256>>>(nblocks, d); break;
    case 4: fold_probe<16, 4><<<1, 512>>>(nblocks, d); break;
    case 5: fold_probe<16, 5><<<1, 512>>>(nblocks, d); break;
    case 6: fold_probe<16, 6><<<1, 512>>>(nblocks, d); break;
    default: fold_probe<16, 7><<<1, 512>>>(nblocks, d); break;
  }
  unsigned long long h[64] = {};
  const cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost);
  cudaFree(d);
  if (e != cudaSuccess) return -1.0;
  double sum = 0;
  for (int w = 0; w < nw; ++w) sum += static_cast<double>(h[w]);
  return sum / nw;
}


// Fold cycles per block of the warps beside the MMA issuer and the copy issuer
// (SM sub-partitions 0 and 1) and of the others (fold_mma_probe): out2[0] = mean
// of warps 4, 5, 8, 9; out2[1] = mean of warps 6, 7, 10, 11.  0 on success.
int w4a4_probe_fold_mma(int nblocks, int mma_per, int tma_per, double* out2) {
  if (nblocks < 1 || nblocks > 100000 || mma_per < 0 || mma_per > 8 || tma_per < 0 || tma_per > 4) return -1;
  unsigned long long* d = nullptr;
  int* status = nullptr;
  uint8_t* g = nullptr;
  if (cudaMalloc(&d, 64 * sizeof(unsigned long long)) != cudaSuccess) return -1;
  if (cudaMalloc(&status, sizeof(int)) != cudaSuccess) { cudaFree(d); return -1; }
  if (cudaMalloc(&g, size_t(4096) * 4096 + 4096) != cudaSuccess) { cudaFree(d); cudaFree(status); return -1; }
  cudaMemset(d, 0, 64 * sizeof(unsigned long long));
  cudaMemset(status, 0, sizeof(int));
  const size_t smem = 48 * 1024;
  cudaFuncSetAttribute(fold_mma_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  fold_mma_probe<<<1, 384, smem>>>(nblocks, mma_per, tma_per, g, d, status);
  unsigned long long h[64] = {};
  int hs = 1;
  const cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) {
    cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost);
    cudaMemcpy(&hs, status, sizeof(int), cudaMemcpyDeviceToHost);
  }
  cudaFree(d);
  cudaFree(status);
  cudaFree(g);
  if (e != cudaSuccess || hs != 0) return -1;
  out2[0] = (h[4] + h[5] + h[8] + h[9]) / 4.0;
  out2[1] = (h[6] + h[7] + h[10] + h[11]) / 4.0;
  return 0;
}

}  // extern "C"
