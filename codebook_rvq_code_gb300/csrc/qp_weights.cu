// Load-time weight preparation: pack caller matrices into the tensor-core
// slice layout, and precompute the squared norm of every embedding row.
//
// Packed layout of a matrix [N, K] (N, K multiples of 128): 128-row tiles;
// inside a tile the element (row r, column k) sits at
//   (k / 8) * 1024 + (r / 8) * 64 + (r % 8) * 8 + (k % 8)
// i.e. K-major core matrices of 8 rows x 8 values (16 bytes as f16), the
// image a no-swizzle tcgen05 shared-memory descriptor reads with a leading
// (K) byte offset of 16 * 128 and a stride (M) byte offset of 128.  One
// 128-row x 128-column slice is therefore a contiguous run.  Q8_0 keeps the
// same element order with one byte per value; its f16 scales are stored
// [tile][K/128][4 blocks of 32][128 rows].
#include "qp_common.cuh"
#include "qp_internal.h"

namespace qp {

namespace {

__device__ __forceinline__ size_t packed_off(int n, int k, int K) {
  const int mt = n / kTileM, r = n % kTileM;
  return size_t(mt) * K * kTileM + size_t(k >> 3) * (kTileM * 8) + (r >> 3) * 64 + (r & 7) * 8 + (k & 7);
}

// 16-bit rows -> f16 packed: f16 sources are copied, bf16 sources
// converted (exact for values in f16's normal range).
__global__ void k_pack_bf16(const uint16_t* __restrict__ src, int rows, int K, uint16_t* __restrict__ dst,
                            int row0, bool src_f16) {
  const size_t total = size_t(rows) * (K / 8);
  for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < total; i += size_t(gridDim.x) * blockDim.x) {
    const int r = int(i / (K / 8)), k8 = int(i % (K / 8));
    const uint4 v = *reinterpret_cast<const uint4*>(src + size_t(r) * K + k8 * 8);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      o[j] = src_f16 ? w[j]
                     : uint32_t(f32_to_f16_bits(bf16_bits_to_f32(w[j] & 0xffff))) |
                           (uint32_t(f32_to_f16_bits(bf16_bits_to_f32(w[j] >> 16))) << 16);
    *reinterpret_cast<uint4*>(dst + packed_off(row0 + r, k8 * 8, K)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Q8_0 block stream rows ({f16 d; int8 q[32]} per 32 values) -> packed int8
// values plus packed scales.  One thread per block.
__global__ void k_pack_q8(const uint8_t* __restrict__ src, int rows, int K, int8_t* __restrict__ dq,
                          __half* __restrict__ ds, int row0) {
  const int nb = K / 32;
  const size_t total = size_t(rows) * nb;
  for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < total; i += size_t(gridDim.x) * blockDim.x) {
    const int r = int(i / nb), kb = int(i % nb);
    const uint8_t* b = src + i * 34;
    const int n = row0 + r;
    const int mt = n / kTileM, rr = n % kTileM, k = kb * 32;
    ds[(size_t(mt) * (K / kKs) + k / kKs) * (kKs / 32) * kTileM + ((k % kKs) / 32) * kTileM + rr] =
        __ushort_as_half(static_cast<unsigned short>(b[0] | (b[1] << 8)));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        lo |= uint32_t(b[2 + j * 8 + e]) << (8 * e);
        hi |= uint32_t(b[2 + j * 8 + 4 + e]) << (8 * e);
      }
      *reinterpret_cast<uint2*>(dq + packed_off(n, k + j * 8, K)) = make_uint2(lo, hi);
    }
  }
}

// Q8_0 block stream rows -> the f16 images hi = f16(d * q) and lo =
// f16(d * q - hi) in the 16-bit packed layout.  d * q is exact in f32 (an
// 11-bit times an 8-bit significand) and so is d * q - hi; lo holds it
// exactly whenever d >= 2^-14 (it is a multiple of d's last place and below
// half of hi's), so hi + lo is the stored weight.  One thread per 8 values.
__global__ void k_pack_q8_hilo(const uint8_t* __restrict__ src, int rows, int K, uint16_t* __restrict__ hi,
                               uint16_t* __restrict__ lo, int row0) {
  const size_t total = size_t(rows) * (K / 8);
  for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < total; i += size_t(gridDim.x) * blockDim.x) {
    const int r = int(i / (K / 8)), k8 = int(i % (K / 8)), k = k8 * 8;
    const uint8_t* b = src + (size_t(r) * (K / 32) + k / 32) * 34;
    const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(b[0] | (b[1] << 8))));
    uint32_t oh[4], ol[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t wh = 0, wl = 0;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float v = d * float(static_cast<int8_t>(b[2 + (k % 32) + 2 * j + e]));
        const __half h = __float2half_rn(v);
        const __half l = __float2half_rn(v - __half2float(h));
        wh |= uint32_t(__half_as_ushort(h)) << (16 * e);
        wl |= uint32_t(__half_as_ushort(l)) << (16 * e);
      }
      oh[j] = wh; ol[j] = wl;
    }
    const size_t o = packed_off(row0 + r, k, K);
    *reinterpret_cast<uint4*>(hi + o) = make_uint4(oh[0], oh[1], oh[2], oh[3]);
    *reinterpret_cast<uint4*>(lo + o) = make_uint4(ol[0], ol[1], ol[2], ol[3]);
  }
}

__global__ void k_row_sumsq(const uint16_t* __restrict__ E, int cols, float* __restrict__ out, bool f16) {
  __shared__ float red[32];
  const uint16_t* row = E + size_t(blockIdx.x) * cols;
  float s = 0.f;
  for (int i = threadIdx.x; i < cols; i += blockDim.x) {
    const float v = e16_to_f32(row[i], f16);
    s += v * v;
  }
  s = block_sum(s, red);
  if (threadIdx.x == 0) out[blockIdx.x] = s;
}

// out[b][j][:] = E_j[codes[b][j]][:] (f16 or bf16 -> f32, exact), 4 values a thread.
struct EmbTables {
  const uint16_t* t[kMaxSteps];
};

// One warp per output row (frame b, table j): the row's code once, then all
// of a lane's pieces of the table row loaded before any of its stores.
__global__ void k_code_embeddings(EmbTables tabs, int n_tables, int V, int d, const int32_t* __restrict__ codes,
                                  long long rows, float* __restrict__ out, int* status, bool f16) {
  const int lane = threadIdx.x & 31;
  const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long row = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5; row < rows; row += nw) {
    const int j = int(row % n_tables);
    int code = codes[row];
    if (code < 0 || code >= V) {
      if (lane == 0) set_status(status, QP_ERR_BAD_TOKEN);
      code = code < 0 ? 0 : V - 1;
    }
    const uint16_t* src = tabs.t[j] + size_t(code) * d;
    float* dst = out + row * d;
    constexpr int kG = 8;   // 1024 columns per pass
    for (int c0 = lane * 4; c0 < d; c0 += 128 * kG) {
      uint2 e[kG];
#pragma unroll
      for (int i = 0; i < kG; ++i)
        e[i] = c0 + i * 128 < d ? __ldg(reinterpret_cast<const uint2*>(src + c0 + i * 128)) : make_uint2(0, 0);
#pragma unroll
      for (int i = 0; i < kG; ++i) {
        if (c0 + i * 128 >= d) break;
        *reinterpret_cast<float4*>(dst + c0 + i * 128) =
            make_float4(e16_to_f32(e[i].x, f16), e16_to_f32(e[i].x >> 16, f16), e16_to_f32(e[i].y, f16),
                        e16_to_f32(e[i].y >> 16, f16));
      }
    }
  }
}

int grid_for(size_t total) { return int(total / 256 + 1 < 8192 ? total / 256 + 1 : 8192); }

}  // namespace

size_t packed_bytes(int fmt, int N, int K) {
  if (fmt == WF_BF16) return size_t(N) * K * 2;
  return size_t(N) * K + size_t(N) * (K / 32) * 2;
}

cudaError_t pack_rows(const void* src, int fmt, bool src_f16, int rows, int K, const PackedMat& dst, int row0,
                      cudaStream_t s) {
  if (fmt == WF_BF16) {
    k_pack_bf16<<<grid_for(size_t(rows) * (K / 8)), 256, 0, s>>>(static_cast<const uint16_t*>(src), rows, K,
                                                                  reinterpret_cast<uint16_t*>(dst.w), row0, src_f16);
  } else {
    k_pack_q8<<<grid_for(size_t(rows) * (K / 32)), 256, 0, s>>>(static_cast<const uint8_t*>(src), rows, K,
                                                                 reinterpret_cast<int8_t*>(dst.w), dst.scale, row0);
    if (dst.w16[0])
      k_pack_q8_hilo<<<grid_for(size_t(rows) * (K / 8)), 256, 0, s>>>(
          static_cast<const uint8_t*>(src), rows, K, reinterpret_cast<uint16_t*>(dst.w16[0]),
          reinterpret_cast<uint16_t*>(dst.w16[1]), row0);
  }
  return cudaGetLastError();
}

cudaError_t code_embeddings(const uint16_t* const* tables, int n_tables, int V, int d, const int32_t* codes, int B,
                            float* out, int* status, bool f16, cudaStream_t s) {
  if (n_tables < 1 || n_tables > kMaxSteps) return cudaErrorInvalidValue;
  EmbTables tabs{};
  for (int j = 0; j < n_tables; ++j) tabs.t[j] = tables[j];
  const long long rows = (long long)B * n_tables;
  const long long blocks = (rows + 7) / 8;   // 8 warps of 256 threads, a row each
  k_code_embeddings<<<int(blocks < 8192 ? blocks : 8192), 256, 0, s>>>(tabs, n_tables, V, d, codes, rows, out, status,
                                                                       f16);
  return cudaGetLastError();
}

cudaError_t row_sumsq_e16(const uint16_t* E, int rows, int cols, bool f16, float* out, cudaStream_t s) {
  k_row_sumsq<<<rows, 256, 0, s>>>(E, cols, out, f16);
  return cudaGetLastError();
}

}  // namespace qp
