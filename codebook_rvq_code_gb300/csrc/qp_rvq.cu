// RVQ codebook normalisation and decode: include/qp_rvq.h.
//
// Both are gathers/streams with no reuse inside one call, so they are plain
// grid-stride kernels moving 16 bytes per thread access: the normalisation
// streams embedding_sum once; the decode reads, per frame, one codebook row
// per stage (the codebooks stay L2-resident at the sizes the codec uses) and
// writes the frame's sum once.  One warp covers 128 consecutive columns of a
// frame, so each codebook row is read as whole 512-byte runs.
#include "qp_common.cuh"
#include "qp_internal.h"
#include "../../include/qp_rvq.h"

namespace qp {
namespace {

constexpr int kRvqMaxCodebooks = 32;   // the decode broadcasts a frame's codes across one warp

__global__ void k_rvq_normalize(const float4* __restrict__ es, const float* __restrict__ usage, long long rows,
                                int d4, float4* __restrict__ out) {
  const long long total = rows * d4;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const float den = __fadd_rn(usage[i / d4], 1e-7f);
    const float4 v = es[i];
    out[i] = make_float4(__fdiv_rn(v.x, den), __fdiv_rn(v.y, den), __fdiv_rn(v.z, den), __fdiv_rn(v.w, den));
  }
}

__global__ void k_rvq_decode(const float* __restrict__ cb, int Q, int K, int D, const int32_t* __restrict__ codes,
                             long long N, float* __restrict__ out, int* status) {
  const int lane = threadIdx.x & 31;
  const int chunks = (D + 127) / 128;
  const long long items = N * chunks;
  const long long warps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long it = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5; it < items; it += warps) {
    const long long n = it / chunks;
    const int d = int(it % chunks) * 128 + lane * 4;
    int code = 0;
    if (lane < Q) {
      code = codes[n * Q + lane];
      if (code < 0 || code >= K) {
        set_status(status, QP_ERR_BAD_TOKEN);
        code = code < 0 ? 0 : K - 1;
      }
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    // stages in order; eight rows in flight at a time
    for (int q0 = 0; q0 < Q; q0 += 8) {
      float4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int cq = __shfl_sync(0xffffffffu, code, (q0 + j) & 31);   // every lane takes part
        v[j] = (q0 + j < Q && d < D) ? __ldg(reinterpret_cast<const float4*>(cb + (size_t(q0 + j) * K + cq) * D + d))
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (q0 + j < Q) {
          acc.x = __fadd_rn(acc.x, v[j].x);
          acc.y = __fadd_rn(acc.y, v[j].y);
          acc.z = __fadd_rn(acc.z, v[j].z);
          acc.w = __fadd_rn(acc.w, v[j].w);
        }
      }
    }
    if (d < D) *reinterpret_cast<float4*>(out + n * D + d) = acc;
  }
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int grid_of(long long work_items, int threads) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 132;
  const long long want = (work_items + threads - 1) / threads;
  const long long cap = (long long)sms * 8;
  return int(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace
}  // namespace qp

extern "C" {

qp_status qp_rvq_normalize(const float* embedding_sum, const float* cluster_usage, int n_codebooks,
                           int codebook_size, int dim, float* codebooks, qp_stream stream) {
  if (!embedding_sum || !cluster_usage || !codebooks) return QP_ERR_ARG;
  if (n_codebooks <= 0 || codebook_size <= 0 || dim <= 0 || dim % 4) return QP_ERR_ARG;
  if (!qp::al16(embedding_sum) || !qp::al16(codebooks) || (reinterpret_cast<uintptr_t>(cluster_usage) & 3))
    return QP_ERR_ARG;
  const long long rows = (long long)n_codebooks * codebook_size;
  qp::k_rvq_normalize<<<qp::grid_of(rows * (dim / 4), 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const float4*>(embedding_sum), cluster_usage, rows, dim / 4,
      reinterpret_cast<float4*>(codebooks));
  if (cudaGetLastError() != cudaSuccess) return QP_ERR_CUDA;
  return QP_OK;
}

qp_status qp_rvq_decode(const float* codebooks, int n_codebooks, int codebook_size, int dim,
                        const int32_t* codes, int n_frames, float* out, int* status, qp_stream stream) {
  if (n_frames < 0 || n_codebooks <= 0 || n_codebooks > qp::kRvqMaxCodebooks || codebook_size <= 0 || dim <= 0 ||
      dim % 4)
    return QP_ERR_ARG;
  if (n_frames == 0) return QP_OK;
  if (!codebooks || !codes || !out || !qp::al16(codebooks) || !qp::al16(out) ||
      (reinterpret_cast<uintptr_t>(codes) & 3))
    return QP_ERR_ARG;
  const long long warps = (long long)n_frames * ((dim + 127) / 128);
  qp::k_rvq_decode<<<qp::grid_of(warps * 32, 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      codebooks, n_codebooks, codebook_size, dim, codes, n_frames, out, status);
  if (cudaGetLastError() != cudaSuccess) return QP_ERR_CUDA;
  return QP_OK;
}

}  // extern "C"
