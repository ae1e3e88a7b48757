// Device helpers shared by the library's kernels.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace qp {

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ float f16_bits_to_f32(uint16_t b) { return __half2float(__ushort_as_half(b)); }

__device__ __forceinline__ uint16_t f32_to_f16_bits(float f) { return __half_as_ushort(__float2half_rn(f)); }
// One element of a 16-bit embedding table, stored as f16 or as bf16 (low 16 bits of b).
__device__ __forceinline__ float e16_to_f32(uint32_t b, bool f16) {
  return f16 ? f16_bits_to_f32(uint16_t(b & 0xffff)) : bf16_bits_to_f32(b & 0xffff);
}

// The f16 tensor-core operand of a Q8_0 weight: d * q rounded once to f16.
__device__ __forceinline__ float q8_0_operand(float d, int q) { return __half2float(__float2half_rn(d * float(q))); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// Sum over the block; every thread gets the result.  red must hold 32 floats.
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float t = lane < nw ? red[lane] : 0.f;
  return warp_sum(t);
}

// Order-preserving map of an f32 to u32 (larger float -> larger key).
__device__ __forceinline__ uint32_t f32_order_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Packed (value, index) for a max-reduction that prefers the lowest index.
__device__ __forceinline__ unsigned long long pack_argmax(float v, int idx) {
  return (static_cast<unsigned long long>(f32_order_key(v)) << 32) |
         static_cast<unsigned long long>(0xffffffffu - static_cast<uint32_t>(idx));
}
__device__ __forceinline__ int unpack_argmax_index(unsigned long long p) {
  return static_cast<int>(0xffffffffu - static_cast<uint32_t>(p & 0xffffffffull));
}

// Latch the first device-detected error into the status word.
__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.f + expf(-z)); }

}  // namespace qp
