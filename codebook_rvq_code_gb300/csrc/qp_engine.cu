// The Code Predictor frame loop as a sequence of per-operation kernels.
//
// One call runs, for B frames at once:
//   step 1: positions 0 = small_to_mtp(H) and 1 = small_to_mtp(E0[q0]);
//   step k: position k = E[k-2][q_{k-1}] for k >= 2;
//   every position: 5 decoder layers (RMSNorm -> fused QKV -> per-head
//   QK-RMSNorm + RoPE -> causal GQA attention over positions 0..k ->
//   O-proj + residual -> RMSNorm -> gate/up -> SwiGLU -> down + residual);
//   then output RMSNorm, lm_head[k-1], and the greedy or Gumbel top-k
//   decision, whose code selects the next position's embedding row.
// ("テキスト音声合成モデルを50ミリ秒未満で応答させる方法", "Qwen3-TTSの最適化方法"
// item 3: 15 fixed steps with a preallocated KV cache; "rightkit-qts 0.2.3",
// "Loader contract": the block tensors and geometry.)
#include <cstdio>

#include "qp_common.cuh"
#include "qp_internal.h"

namespace qp {

namespace {

enum GemmMode { G_STORE = 0, G_ADD = 1, G_STORE_BIAS = 2 };

template <int FMT>
__device__ __forceinline__ float load_w(const QMat& W, int n, int k) {
  if (FMT == WF_BF16) {
    return bf16_bits_to_f32(static_cast<const uint16_t*>(W.w)[size_t(n) * W.K + k]);
  } else {
    const float d = __half2float(W.scale[size_t(n) * (W.K / 32) + (k >> 5)]);
    return q8_0_operand(d, static_cast<const int8_t*>(W.w)[size_t(n) * W.K + k]);
  }
}

// C[m, n] (=, +=, = .. + bias[n]) sum_k A[m, k] * W[n, k]; A f16 [M, lda].
// Tiles of 32 rows x 64 outputs x 32 k; N % 64 == 0, K % 32 == 0.
template <int FMT>
__global__ void __launch_bounds__(256) k_gemm_tiled(const uint16_t* __restrict__ A, int lda, int M, QMat W,
                                                    float* __restrict__ C, int ldc,
                                                    const float* __restrict__ bias, int mode) {
  constexpr int BM = 32, BN = 64, BK = 32;
  __shared__ float As[BK][BM + 1];
  __shared__ float Ws[BK][BN + 1];
  const int tid = threadIdx.x;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int tx = tid & 15, ty = tid >> 4;
  float acc[2][4] = {};
  for (int k0 = 0; k0 < W.K; k0 += BK) {
    {
      const int r = tid >> 3, kk = (tid & 7) * 4, m = m0 + r;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        As[kk + j][r] = m < M ? f16_bits_to_f32(A[size_t(m) * lda + k0 + kk + j]) : 0.f;
    }
    {
      const int r = tid >> 2, kk = (tid & 3) * 8, n = n0 + r;
#pragma unroll
      for (int j = 0; j < 8; ++j) Ws[kk + j][r] = load_w<FMT>(W, n, k0 + kk + j);
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < BK; ++kk) {
      const float a0 = As[kk][ty * 2], a1 = As[kk][ty * 2 + 1];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float w = Ws[kk][tx * 4 + j];
        acc[0][j] = fmaf(a0, w, acc[0][j]);
        acc[1][j] = fmaf(a1, w, acc[1][j]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int m = m0 + ty * 2 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      float* c = C + size_t(m) * ldc + n;
      if (mode == G_ADD) *c += acc[i][j];
      else if (mode == G_STORE_BIAS) *c = acc[i][j] + bias[n];
      else *c = acc[i][j];
    }
  }
}

// act rows 2b = f16(H[b]), 2b+1 = f16(E0[q0[b]]) (the two inputs of step 1).
__global__ void k_prepare_inputs(const float* __restrict__ H, const int32_t* __restrict__ q0,
                                 const uint16_t* __restrict__ e0, int th, int q0_vocab,
                                 uint16_t* __restrict__ act, int* status) {
  const int r = blockIdx.x, b = r >> 1;
  uint16_t* dst = act + size_t(r) * th;
  if ((r & 1) == 0) {
    for (int i = threadIdx.x; i < th; i += blockDim.x) dst[i] = f32_to_f16_bits(H[size_t(b) * th + i]);
  } else {
    int q = q0[b];
    if (q < 0 || q >= q0_vocab) {
      if (threadIdx.x == 0) set_status(status, QP_ERR_BAD_TOKEN);
      q = q < 0 ? 0 : q0_vocab - 1;
    }
    for (int i = threadIdx.x; i < th; i += blockDim.x)
      dst[i] = f32_to_f16_bits(bf16_bits_to_f32(e0[size_t(q) * th + i]));
  }
}

// act[r] = f16(RMSNorm(src[r * stride]) * w), d columns.
__global__ void k_rmsnorm(const float* __restrict__ src, int stride, int d, const float* __restrict__ w,
                          float eps, uint16_t* __restrict__ act) {
  __shared__ float red[32];
  const float* x = src + size_t(blockIdx.x) * stride;
  float ss = 0.f;
  for (int i = threadIdx.x; i < d; i += blockDim.x) ss += x[i] * x[i];
  ss = block_sum(ss, red);
  const float inv = rsqrtf(ss / float(d) + eps);
  for (int i = threadIdx.x; i < d; i += blockDim.x)
    act[size_t(blockIdx.x) * d + i] = f32_to_f16_bits(x[i] * inv * w[i]);
}

// Per-head RMSNorm then rotate-half RoPE of a 128-vector held one element per
// thread (blockDim.x == 128).
__device__ __forceinline__ float head_norm_rope(float v, const float* __restrict__ nw, float eps,
                                                const float2* __restrict__ cs_row, float* xs, float* red) {
  const int t = threadIdx.x;
  const float ss = block_sum(v * v, red);
  const float n = v * rsqrtf(ss / 128.f + eps) * nw[t];
  xs[t] = n;
  __syncthreads();
  const float2 cs = cs_row[t & 63];
  const float r = t < 64 ? n * cs.x - xs[t + 64] * cs.y : n * cs.x + xs[t - 64] * cs.y;
  __syncthreads();
  return r;
}

// Attention for one frame and one kv head over the new position(s).
// grid (B, n_kv), block 128.  kv layout [b][pos][2][n_kv][128] (this layer).
__global__ void __launch_bounds__(128) k_attention(const float* __restrict__ qkv, int ld, int P, int pos0,
                                                   float* __restrict__ kv, int ctx, int n_q, int n_kv,
                                                   const float* __restrict__ q_norm,
                                                   const float* __restrict__ k_norm,
                                                   const float2* __restrict__ rope_cs, float eps,
                                                   uint16_t* __restrict__ act) {
  __shared__ float red[32];
  __shared__ float xs[128];
  __shared__ float sc[kMaxCtx];
  const int b = blockIdx.x, j = blockIdx.y, t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int qw = n_q * 128, kvw = n_kv * 128, grp = n_q / n_kv;
  float* kvb = kv + size_t(b) * ctx * 2 * kvw;
  for (int p = 0; p < P; ++p) {
    const int r = b * P + p, pos = pos0 + p;
    const float kr = qkv[size_t(r) * ld + qw + j * 128 + t];
    const float ko = head_norm_rope(kr, k_norm, eps, rope_cs + pos * 64, xs, red);
    const float v = qkv[size_t(r) * ld + qw + kvw + j * 128 + t];
    kvb[(size_t(pos) * 2 + 0) * kvw + j * 128 + t] = ko;
    kvb[(size_t(pos) * 2 + 1) * kvw + j * 128 + t] = v;
  }
  __syncthreads();
  const float scale = rsqrtf(128.f);
  for (int p = 0; p < P; ++p) {
    const int r = b * P + p, pos = pos0 + p;
    for (int gi = 0; gi < grp; ++gi) {
      const int hq = j * grp + gi;
      const float qr = qkv[size_t(r) * ld + hq * 128 + t];
      const float qo = head_norm_rope(qr, q_norm, eps, rope_cs + pos * 64, xs, red);
      xs[t] = qo;
      __syncthreads();
      for (int i = warp; i <= pos; i += 4) {
        const float* kr = kvb + (size_t(i) * 2 + 0) * kvw + j * 128;
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) s += xs[lane * 4 + e] * kr[lane * 4 + e];
        s = warp_sum(s);
        if (lane == 0) sc[i] = s * scale;
      }
      __syncthreads();
      float mx = -INFINITY;
      for (int i = 0; i <= pos; ++i) mx = fmaxf(mx, sc[i]);
      float den = 0.f, o = 0.f;
      for (int i = 0; i <= pos; ++i) {
        const float e = expf(sc[i] - mx);
        den += e;
        o += e * kvb[(size_t(i) * 2 + 1) * kvw + j * 128 + t];
      }
      act[size_t(r) * qw + hq * 128 + t] = f32_to_f16_bits(o / den);
      __syncthreads();
    }
  }
}

// act[r, j] = f16(silu(gate[r, j]) * up[r, j]); gu rows = [gate (F) | up (F)].
__global__ void k_swiglu(const float* __restrict__ gu, int M, int F, uint16_t* __restrict__ act) {
  const size_t n = size_t(M) * F;
  for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < n; i += size_t(gridDim.x) * blockDim.x) {
    const size_t r = i / F, c = i % F;
    const float gt = gu[r * 2 * F + c], up = gu[r * 2 * F + F + c];
    act[i] = f32_to_f16_bits(silu_f(gt) * up);
  }
}

// Decision of step `step` (1-based) for frame blockIdx.x: greedy argmax, or
// Gumbel-max over the top-k of logits/T.  Writes the code, optionally the
// logits, and the next position's input row X[b] = E[step-1][next code].
constexpr int kDecideThreads = 256;
constexpr int kMaxVocab = 8192;

__global__ void __launch_bounds__(kDecideThreads) k_decide(
    const float* __restrict__ logits, int V, int step, int n_steps, float temperature, int top_k,
    const float* __restrict__ gumbel, const int32_t* __restrict__ forced, int32_t* __restrict__ out_codes,
    float* __restrict__ out_logits, const uint16_t* __restrict__ next_embed, float* __restrict__ X, int d,
    int* status) {
  __shared__ unsigned long long redu[32];
  __shared__ int sh_code;
  const int b = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const float* l = logits + size_t(b) * V;
  if (out_logits) {
    float* o = out_logits + (size_t(b) * n_steps + (step - 1)) * V;
    for (int i = t; i < V; i += kDecideThreads) o[i] = l[i];
  }
  unsigned long long best = 0ull;
  if (temperature <= 0.f) {
    for (int i = t; i < V; i += kDecideThreads) {
      const unsigned long long pk = pack_argmax(l[i], i);
      best = pk > best ? pk : best;
    }
  } else {
    __shared__ uint32_t keys[kMaxVocab];
    __shared__ int hist[256];
    __shared__ int sh_sel, sh_rem;
    __shared__ int chunk_cnt[kDecideThreads];
    for (int i = t; i < V; i += kDecideThreads) keys[i] = f32_order_key(l[i] / temperature);
    uint32_t prefix = 0, mask = 0;
    int remaining = top_k;
    for (int shift = 24; shift >= 0; shift -= 8) {
      hist[t] = 0;
      __syncthreads();
      for (int i = t; i < V; i += kDecideThreads) {
        const uint32_t k = keys[i];
        if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255], 1);
      }
      __syncthreads();
      if (t == 0) {
        int cum = 0, sel = 0;
        for (int dg = 255; dg >= 0; --dg) {
          if (cum + hist[dg] >= remaining) { sel = dg; break; }
          cum += hist[dg];
        }
        sh_sel = sel;
        sh_rem = remaining - cum;
      }
      __syncthreads();
      prefix |= uint32_t(sh_sel) << shift;
      mask |= 255u << shift;
      remaining = sh_rem;
      __syncthreads();
    }
    const uint32_t kth = prefix;
    // rank of each key equal to kth among its equals, by index
    const int per = (V + kDecideThreads - 1) / kDecideThreads;
    const int lo = t * per, hi = min(V, lo + per);
    int cnt = 0;
    for (int i = lo; i < hi; ++i) cnt += keys[i] == kth;
    chunk_cnt[t] = cnt;
    __syncthreads();
    if (t == 0) {
      int run = 0;
      for (int i = 0; i < kDecideThreads; ++i) { const int c = chunk_cnt[i]; chunk_cnt[i] = run; run += c; }
    }
    __syncthreads();
    int eq_rank = chunk_cnt[t];
    const float* gb = gumbel + (size_t(b) * n_steps + (step - 1)) * V;
    for (int i = lo; i < hi; ++i) {
      const uint32_t k = keys[i];
      bool in = k > kth;
      if (k == kth) { in = eq_rank < remaining; ++eq_rank; }
      if (in) {
        const float z = l[i] / temperature;
        const unsigned long long pk = pack_argmax(z + gb[i], i);
        best = pk > best ? pk : best;
      }
    }
  }
  best = warp_max_u64(best);
  if (lane == 0) redu[warp] = best;
  __syncthreads();
  if (warp == 0) {
    unsigned long long v = lane < kDecideThreads / 32 ? redu[lane] : 0ull;
    v = warp_max_u64(v);
    if (lane == 0) {
      const int code = unpack_argmax_index(v);
      out_codes[size_t(b) * n_steps + (step - 1)] = code;
      int nc = forced ? forced[size_t(b) * n_steps + (step - 1)] : code;
      if (nc < 0 || nc >= V) {
        set_status(status, QP_ERR_BAD_TOKEN);
        nc = nc < 0 ? 0 : V - 1;
      }
      sh_code = nc;
    }
  }
  __syncthreads();
  if (next_embed) {
    const uint16_t* e = next_embed + size_t(sh_code) * d;
    for (int i = t; i < d; i += kDecideThreads) X[size_t(b) * d + i] = bf16_bits_to_f32(e[i]);
  }
}

__global__ void k_repack_q8_0(const uint8_t* __restrict__ blocks, int N, int K, int8_t* __restrict__ qs,
                              __half* __restrict__ d) {
  const int nb = K / 32;
  const size_t total = size_t(N) * nb;
  for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < total; i += size_t(gridDim.x) * blockDim.x) {
    const uint8_t* src = blocks + i * 34;
    const unsigned short bits = static_cast<unsigned short>(src[0] | (src[1] << 8));
    d[i] = __ushort_as_half(bits);
    for (int j = 0; j < 32; ++j) qs[i * 32 + j] = static_cast<int8_t>(src[2 + j]);
  }
}

void gemm(const uint16_t* A, int lda, int M, const QMat& W, float* C, int ldc, const float* bias, int mode,
          cudaStream_t s) {
  dim3 grid(W.N / 64, (M + 31) / 32);
  if (W.fmt == WF_BF16)
    k_gemm_tiled<WF_BF16><<<grid, 256, 0, s>>>(A, lda, M, W, C, ldc, bias, mode);
  else
    k_gemm_tiled<WF_Q8_0><<<grid, 256, 0, s>>>(A, lda, M, W, C, ldc, bias, mode);
}

}  // namespace

cudaError_t repack_q8_0(const uint8_t* blocks, int N, int K, int8_t* qs, __half* d, cudaStream_t s) {
  const size_t total = size_t(N) * (K / 32);
  const int grid = int((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
  k_repack_q8_0<<<grid, 256, 0, s>>>(blocks, N, K, qs, d);
  return cudaGetLastError();
}

int launches_per_call(const qp_handle* h, int /*B*/, bool /*sampling*/) {
  return 2 + h->g.n_steps * (h->g.layers * 8 + 3);
}

qp_status run_frames(qp_handle* h, const RunArgs& a, cudaStream_t s) {
  const qp_geometry& g = h->g;
  const int B = a.B, d = g.hidden, qw = g.n_q_heads * 128, kvw = g.n_kv_heads * 128;
  const int qkvw = qw + 2 * kvw, ctx = g.n_steps + 1;
  if (a.temperature > 0.f && g.vocab > kMaxVocab) return QP_ERR_ARG;

  k_prepare_inputs<<<2 * B, 256, 0, s>>>(a.H, a.q0, h->e0, g.talker_hidden, g.q0_vocab, h->act, h->status);
  gemm(h->act, g.talker_hidden, 2 * B, h->proj, h->X, d, h->b_proj, G_STORE_BIAS, s);
  for (int k = 1; k <= g.n_steps; ++k) {
    const int P = k == 1 ? 2 : 1, M = B * P, pos0 = k == 1 ? 0 : k;
    for (int l = 0; l < g.layers; ++l) {
      const LayerW& L = h->layer[l];
      float* kv_l = h->kv + size_t(l) * h->max_batch * ctx * 2 * kvw;
      k_rmsnorm<<<M, 256, 0, s>>>(h->X, d, d, L.attn_norm, g.rms_eps, h->act);
      gemm(h->act, d, M, L.qkv, h->qkv, qkvw, nullptr, G_STORE, s);
      k_attention<<<dim3(B, g.n_kv_heads), 128, 0, s>>>(h->qkv, qkvw, P, pos0, kv_l, ctx, g.n_q_heads,
                                                         g.n_kv_heads, L.q_norm, L.k_norm, h->rope_cs,
                                                         g.rms_eps, h->act);
      gemm(h->act, qw, M, L.o, h->X, d, nullptr, G_ADD, s);
      k_rmsnorm<<<M, 256, 0, s>>>(h->X, d, d, L.ffn_norm, g.rms_eps, h->act);
      gemm(h->act, d, M, L.gu, h->gu, 2 * g.ffn, nullptr, G_STORE, s);
      k_swiglu<<<(M * g.ffn + 255) / 256 < 8192 ? (M * g.ffn + 255) / 256 : 8192, 256, 0, s>>>(h->gu, M, g.ffn,
                                                                                             h->act);
      gemm(h->act, g.ffn, M, L.down, h->X, d, nullptr, G_ADD, s);
    }
    k_rmsnorm<<<B, 256, 0, s>>>(h->X + (P - 1) * d, P * d, d, h->out_norm, g.rms_eps, h->act);
    gemm(h->act, d, B, h->head[k - 1], h->logits, g.vocab, nullptr, G_STORE, s);
    k_decide<<<B, kDecideThreads, 0, s>>>(h->logits, g.vocab, k, g.n_steps, a.temperature, a.top_k, a.gumbel,
                                          a.forced, a.out_codes, a.out_logits,
                                          k < g.n_steps ? h->embed[k - 1] : nullptr, h->X, d, h->status);
  }
  return cudaGetLastError() == cudaSuccess ? QP_OK : QP_ERR_CUDA;
}

}  // namespace qp
