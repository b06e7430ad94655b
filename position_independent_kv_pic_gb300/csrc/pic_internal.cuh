// Internal helpers shared by the CUDA translation units of the PIC library.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pic.h"

namespace pic {

// First device-side error wins; later ones are dropped.
__device__ __forceinline__ void set_err(int32_t* flag, int32_t code) {
  if (flag != nullptr) atomicCAS(flag, 0, code);
}

__host__ __device__ __forceinline__ int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Storage conversions (round to nearest even on the way down).
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Exclusive scan of one int per thread over a block of NT threads (NT <= 1024,
// multiple of 32).  `scratch` holds NT/32 + 1 ints.  Returns the exclusive prefix;
// *total receives the block sum.  Contains __syncthreads.
template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < NT / 32) ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < NT / 32) scratch[lane] = w;  // inclusive warp totals
    if (lane == NT / 32 - 1) scratch[NT / 32] = w;
  }
  __syncthreads();
  int base = (warp > 0) ? scratch[warp - 1] : 0;
  *total = scratch[NT / 32];
  __syncthreads();
  return base + x - v;
}

// RoPE rotation of one dimension pair (a, b) = (x_i, x_{i+d/2}) by an angle
// whose cos / sin come as unevaluated sums of two floats, t = {cos_hi, sin_hi,
// cos_lo, sin_lo} (hi = v rounded to 16 significant bits, lo = fp32(v - hi),
// from fp64):
//   ya = a cos - b sin,   yb = b cos + a sin.
// The hi products are split exactly with FMA (p + e = a * c_hi); the low-order
// terms are added once.  The result carries about 2^-23 relative error plus
// 2^-46 |x|, so rounding it to bf16 lands within one ulp of the exactly
// rounded value even when the pair nearly cancels.  The _rn intrinsics keep
// the compiler from contracting the split.
__device__ __forceinline__ void rope_rotate(float a, float b, float4 t, float& ya, float& yb) {
  const float p1 = __fmul_rn(a, t.x), e1 = __fmaf_rn(a, t.x, -p1);
  const float p2 = __fmul_rn(b, t.y), e2 = __fmaf_rn(b, t.y, -p2);
  const float p3 = __fmul_rn(b, t.x), e3 = __fmaf_rn(b, t.x, -p3);
  const float p4 = __fmul_rn(a, t.y), e4 = __fmaf_rn(a, t.y, -p4);
  const float ca = __fadd_rn(__fsub_rn(e1, e2), __fmaf_rn(a, t.z, -__fmul_rn(b, t.w)));
  const float cb = __fadd_rn(__fadd_rn(e3, e4), __fmaf_rn(b, t.z, __fmul_rn(a, t.w)));
  ya = __fadd_rn(__fsub_rn(p1, p2), ca);
  yb = __fadd_rn(__fadd_rn(p3, p4), cb);
}

// The same rotation for inputs that are bf16 values (8 significant bits).  The
// table's hi parts carry at most 16 significant bits, so a * cos_hi and b * sin_hi
// are exact in fp32 and one rounding of their difference keeps ~2^-24 relative
// error: same guarantee as rope_rotate at half the operations.
__device__ __forceinline__ void rope_rotate_bf16in(float a, float b, float4 t, float& ya, float& yb) {
  const float u = __fmaf_rn(a, t.x, -__fmul_rn(b, t.y));
  const float v = __fmaf_rn(b, t.x, __fmul_rn(a, t.y));
  ya = __fadd_rn(u, __fmaf_rn(a, t.z, -__fmul_rn(b, t.w)));
  yb = __fadd_rn(v, __fmaf_rn(b, t.z, __fmul_rn(a, t.w)));
}

int num_sms_of_current_device();

// The driver's cuTensorMapEncodeTiled, looked up once through the runtime (null if
// the driver lacks it).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Tensor map of a K or V pool viewed as rows of 128 bf16 (one (block, head, slot) key
// row each): one 4-D box [2 row groups][2 column halves][8 rows][64 columns], 128-byte
// swizzle, moves a whole 16-row page into shared memory as 4 swizzle atoms of 1 KB
// (group g, half h at byte g * 2048 + h * 1024; row r's 16-byte chunk c at
// r * 128 + (c ^ r) * 16).  rows must be a multiple of 8.
bool encode_pages(CUtensorMap* map, const void* base, uint64_t rows);

// SIMT attention launcher (attention_simt.cu); arguments as pic_link_attention.
pic_status launch_attention_simt(const void* q, const float* row_table, const int32_t* rows,
                                 const int32_t* row_off, const void* k_pool, const void* v_pool,
                                 int64_t num_blocks, pic_dtype dtype, const pic_link_page* pages,
                                 const int32_t* page_off, int32_t n_req, int64_t n_rows, int32_t Hq,
                                 int32_t Hkv, int32_t d, float scale, void* out, cudaStream_t s);

}  // namespace pic
