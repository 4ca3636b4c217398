// Internal declarations shared by the CUDA translation units of libw4a4.so.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "w4a4_device.cuh"

namespace w4a4 {

// Number of SMs of the current device (cached per device).
int num_sms();

// Routing tables of one MUL_MAT_ID call, carved out of the caller's workspace.
struct Routing {
  int32_t* hdr;        // [4]: nonzero if some id was outside [0, E); segments; tiles; routed rows
  int32_t* offsets;    // [E + 1] first gathered row of each expert
  int4* segs;          // [segments] {first gathered row, expert, rows (<= 256), weight tiles per tile}
  int32_t* seg_tiles;  // [segments + 1] first tile of each segment
  int32_t* perm;       // [M * top_k] gathered row -> pair index t * top_k + s
  uint8_t* gcodes;     // [M * top_k][K/2] activation codes gathered in expert order
  float* gscales;      // [M * top_k][K/32] their scales
  int64_t rows;        // capacity of the gathered arrays (M * top_k)
  uint32_t* sk_count;  // [sk_ctas * 8] stream-K tickets (zeroed by the routing kernel)
  float4* sk_part;     // [2 * sk_ctas] stream-K partial tiles (grp_sk_part_bytes each)
  int sk_ctas;         // the routed GEMM's grid: one CTA per SM of the current device
};

struct RoutingLayout {
  size_t hdr, offsets, segs, seg_tiles, perm, gcodes, gscales, sk_count, sk_part, total;
  int sk_ctas;
};
RoutingLayout routing_layout(int64_t npairs, int E, int64_t K);
Routing routing_in(void* ws, int64_t npairs, int E, int64_t K);

// Fixed routing scratch (for the no-workspace variant of the routed product):
// its size, and the device address of the current device's copy.
constexpr size_t kIdStaticScratchBytes = size_t(64) << 20;
cudaError_t id_static_scratch(void** addr);

// expanded (optional): the offset codes a + 8 as bytes in element order, [M][K]
// (the e4m3 activation operand of the dense GEMM).
cudaError_t launch_act_rotate_quantize(const float* x, int64_t M, int64_t K, int64_t ldx, int rotate,
                                       uint8_t* codes, float* scales, uint8_t* expanded, cudaStream_t stream);
// The exact path's 8-bit activations: int8 codes [M][K] (element order), fp32 scales.
cudaError_t launch_act_rotate_quantize8(const float* x, int64_t M, int64_t K, int64_t ldx, int rotate,
                                        int8_t* codes, float* scales, cudaStream_t stream);
// The packers and the import also write the expanded weight operand (the e4m3
// bytes of q - 8 in element order, [round_up(N, 8)][K], pad rows zero) when
// `expanded` is not null.
cudaError_t launch_pack_q4_0(const void* w, int w_dtype, int64_t N, int64_t K, int64_t ldw, int rotate,
                             uint8_t* codes, uint16_t* scales, int16_t* sums, uint8_t* expanded,
                             cudaStream_t stream);
// Importance-weighted Q4_0 (the converter's imatrix quantisation): imp is a
// device fp32 vector of K per-input-channel importances (unrotated), or null.
cudaError_t launch_pack_q4_0_weighted(const void* w, int w_dtype, int64_t N, int64_t K, int64_t ldw, int rotate,
                                      const float* imp, uint8_t* codes, uint16_t* scales, int16_t* sums,
                                      uint8_t* expanded, cudaStream_t stream);
cudaError_t launch_import_q4_0(const void* blocks, int64_t N, int64_t K, uint8_t* codes, uint16_t* scales,
                               int16_t* sums, uint8_t* expanded, cudaStream_t stream);
// Dense product (P == nullptr) or exact partials (P != nullptr), both operands
// from their codes.  With a workspace of at least gemm_workspace_bytes(M, N, K)
// bytes (16-byte aligned, zero before its first use) the dense product may run a
// stream-K schedule.  w_expanded (optional, the dense product only): the
// pre-expanded weight operand.
cudaError_t launch_gemm_tc(const uint8_t* w_codes, const uint16_t* w_scales, const int16_t* w_sums,
                           const uint8_t* w_expanded, int64_t N, const uint8_t* a_codes, const float* a_scales,
                           int64_t M, int64_t K, float* y, int64_t ldy, int32_t* P, void* ws, size_t ws_bytes,
                           cudaStream_t stream);
size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);
// The exact path (rotated Q4_0 weights x int8 activations, f16 tensor-core
// MMAs): dense product (P == nullptr) or exact partials; workspace as above.
cudaError_t launch_gemm_w4a8(const uint8_t* w_codes, const uint16_t* w_scales, const int16_t* w_sums, int64_t N,
                             const int8_t* a_codes, const float* a_scales, int64_t M, int64_t K, float* y, int64_t ldy,
                             int32_t* P, void* ws, size_t ws_bytes, cudaStream_t stream);
size_t gemm_w4a8_workspace_bytes(int64_t M, int64_t N, int64_t K);
// The rotate-only route: activations rotated and carried as bf16 [M][K] (not
// quantised), bf16 tensor-core MMAs against the Q4_0 weights; its workspace
// plan is the exact path's (gemm_w4a8_workspace_bytes).
cudaError_t launch_act_rotate_bf16(const float* x, int64_t M, int64_t K, int64_t ldx, int rotate, uint16_t* out,
                                   cudaStream_t stream);
cudaError_t launch_gemm_w4a16(const uint8_t* w_codes, const uint16_t* w_scales, const int16_t* w_sums, int64_t N,
                              const uint16_t* a_bf16, int64_t M, int64_t K, float* y, int64_t ldy, void* ws,
                              size_t ws_bytes, cudaStream_t stream);
// Small token batches (1 <= M <= 8): CUDA-core kernel, bit-identical to the
// tensor-core kernel's whole-tile schedule.
cudaError_t launch_gemm_small_m(const uint8_t* w_codes, const uint16_t* w_scales, int64_t N, const uint8_t* a_codes,
                                const float* a_scales, int M, int64_t K, float* y, int64_t ldy, cudaStream_t stream);
// The super-tile GEMM (gemm_grp.cu).  Dense: expanded activations [round_up(M, 8)][K]
// (offset-code bytes), optional expanded weights; workspace as for launch_gemm_tc,
// of grp_workspace_bytes(M, N, K) bytes.  Routed: the gathered codes and work list
// of `r`, weights as Q4_0 codes.
cudaError_t launch_gemm_grp(const uint8_t* w_codes, const uint16_t* w_scales, const int16_t* w_sums,
                            const uint8_t* w_expanded, int64_t N, const uint8_t* a_expanded, const float* a_scales,
                            int64_t M, int64_t K, float* y, int64_t ldy, void* ws, size_t ws_bytes,
                            cudaStream_t stream);
size_t grp_workspace_bytes(int64_t M, int64_t N, int64_t K);
// Bytes of one stream-K partial tile of the super-tile kernel (8 warps x 32 lanes x
// 128 accumulators); a CTA needs two.
size_t grp_sk_part_bytes();
cudaError_t launch_gemm_grp_routed(const uint8_t* w_codes, const uint16_t* w_scales, const int16_t* w_sums,
                                   int E, int64_t N, int64_t K, const Routing& r, float* y, cudaStream_t stream);
// Test hook: the bound of the super-tile GEMM's pipeline waits (0 = the default
// second) and a delay before its producer's first copy.
void grp_set_wait_limit(uint64_t wait_ns, uint64_t producer_delay_ns);
// Reads the GEMM kernels' device error word (bounded waits that gave up) and clears it.
cudaError_t read_and_clear_device_error(int* value);
// Device address of the error word the GEMM and activation kernels set when a
// bounded wait gives up (nullptr on failure).
int* device_error_word();
// 2D tiled TMA descriptor over `rows` rows of `inner` elements.
cudaError_t encode_2d_map(CUtensorMap* m, CUtensorMapDataType dtype, const void* base, uint64_t inner, uint64_t rows,
                          uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle);
cudaError_t launch_gemm_id(const uint8_t* w_codes, const uint16_t* w_scales, const int16_t* w_sums, int E,
                           int64_t N, const uint8_t* a_codes, const float* a_scales, int64_t K, const int32_t* ids,
                           int64_t M, int top_k, int act_per_slot, float* y, const Routing& r, cudaStream_t stream);

}  // namespace w4a4
