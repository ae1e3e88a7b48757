// The Code Predictor frame loop as ONE persistent cooperative kernel.
//
// The whole 15-step loop of a batch of frames ("テキスト音声合成モデルを50ミリ秒未満で
// 応答させる方法", "Qwen3-TTSの最適化方法" item 3: a fixed GPU program in place
// of a host-driven sequence, with a preallocated KV cache) runs as a list of
// phases separated by grid barriers.  Every weight contraction is a GEMM
// phase on the tcgen05 tensor cores:
//
//   D[128 weight rows, Nc rows of frames] += W[128, K-slice] * act[Nc, K-slice]^T
//
// with f16 operands and an f32 accumulator in TMEM.  Weights are packed at
// load time into exactly the shared-memory image the MMA descriptors read
// (K-major 8x16-byte core matrices, no swizzle), so one K-slice of one
// 128-row tile is one contiguous cp.async.bulk.  A producer warp streams the
// CTA's weight slices for all phases, in order, through a ring of shared
// memory slots; it never waits on the grid, so weight traffic runs ahead
// across phase boundaries.  GEMM slices are dealt out to CTAs in equal
// contiguous runs (stream-K style); each run's partial tile is added into an
// f32 accumulator in global memory with red.add.  Elementwise phases (RMSNorm,
// QK-norm + RoPE + attention, SwiGLU, the decision) run on the same CTAs.
#include <cooperative_groups.h>
#include <cstdio>

#include "qp_common.cuh"
#include "qp_internal.h"
#include "qp_ptx.cuh"

namespace qp {

namespace {

constexpr int kConsumers = 256;             // 8 consumer warps
constexpr int kThreads = kConsumers + 32;   // + 1 producer warp
constexpr int kNSlot = 4;                   // weight ring slots
constexpr int kKs = 128;                    // K per slice
constexpr int kTileM = 128;                 // weight rows per MMA tile
constexpr int kMaxNc = 128;                 // frames per MMA (N)
constexpr uint32_t kSlotBytes = kTileM * kKs * 2;          // 32 KB f16
constexpr uint32_t kQ8Bytes = kTileM * kKs;                // 16 KB int8
constexpr uint32_t kQ8ScaleBytes = (kKs / 32) * kTileM * 2;  // 1 KB f16
constexpr uint32_t kActBytes = kKs * kMaxNc * 2;           // 32 KB
constexpr uint32_t kTmemCols = 128;

enum { BAR_ALL = 1, BAR_H0 = 2, BAR_H1 = 3 };

struct PLayer {
  const uint8_t* w_qkv; const __half* s_qkv;
  const uint8_t* w_o; const __half* s_o;
  const uint8_t* w_gu; const __half* s_gu;
  const uint8_t* w_d; const __half* s_d;
  const float* attn_norm; const float* q_norm; const float* k_norm; const float* ffn_norm;
};

struct PParams {
  int d, qw, kvw, F, V, th, L, n_q, n_kv, n_steps, q0_vocab;
  float eps;
  int q8;
  const uint8_t* w_proj; const __half* s_proj; const float* b_proj;
  const uint16_t* e0;
  PLayer layer[kMaxLayers];
  const float* out_norm;
  const uint16_t* embed[kMaxSteps];
  const uint8_t* w_head[kMaxSteps]; const __half* s_head[kMaxSteps];
  const float2* rope_cs;
  float* xres; uint16_t* act; float* acc_qkv; float* acc_gu; float* logits; float* kv;
  unsigned int* bar; int* abort_flag; int* status;
  int Bmax;
  int B; const float* H; const int32_t* q0; int32_t* out_codes; float* out_logits; const int32_t* forced;
  float temperature; int top_k; const float* gumbel;
};

struct Smem {
  alignas(1024) uint8_t slot[kNSlot][kSlotBytes];
  alignas(1024) uint8_t actb[kActBytes];
  union {   // the Q8_0 operand in GEMM phases, the top-k keys in the decision
    alignas(1024) uint8_t deq[kSlotBytes];
    uint32_t keys[8192];
  };
  alignas(8) uint64_t full[kNSlot];
  alignas(8) uint64_t empty[kNSlot];
  alignas(8) uint64_t actbar;
  alignas(8) uint64_t mmabar;
  uint32_t tmem_base;
  float red[2][8];
  float xs[2][128];
  float sc[2][kMaxCtx];
  unsigned long long redu[8];
  int sh_int[8];
  int hist[256];
  int chunk_cnt[kConsumers];
};

// N-chunking of R rows for the MMA: chunks of Nc (multiple of 16, <= 128).
struct Chunking { int Nc, n_chunks; };
__device__ __forceinline__ Chunking chunking(int R) {
  const int r16 = (R + 15) & ~15;
  if (r16 <= kMaxNc) return {r16, 1};
  return {kMaxNc, (R + kMaxNc - 1) / kMaxNc};
}

// Element offset of (row n, feature k) in the activation operand layout
// [chunk][K/8][Nc/8][8 rows][8 k] for reduction length Kdim.
__device__ __forceinline__ size_t act_off(int n, int k, int Kdim, Chunking c) {
  const int ch = n / c.Nc, nn = n - ch * c.Nc;
  return size_t(ch) * Kdim * c.Nc + (size_t((k >> 3) * (c.Nc >> 3) + (nn >> 3)) << 6) + ((nn & 7) << 3) + (k & 7);
}

struct Gemm {
  const uint8_t* w; const __half* s;
  int n_mt, n_ks;       // 128-row tiles, 128-wide K slices
  int Kdim;
  float* acc; int ld;   // acc[row][feature]
  int R;
};

// The CTA's contiguous run [beg, end) of the phase's slices.
__device__ __forceinline__ void my_slices(int total, int gemm_idx, int& beg, int& end) {
  const int G = gridDim.x;
  const int g = (blockIdx.x + gemm_idx * 37) % G;
  beg = int((long long)total * g / G);
  end = int((long long)total * (g + 1) / G);
}

// ---------------------------------------------------------------------------
// The phase program.  Producer and consumers walk the same sequence of GEMM
// phases; this builds the i-th one (call order) for both.
// ---------------------------------------------------------------------------
struct Prog {
  const PParams& p;
  __device__ Prog(const PParams& pp) : p(pp) {}
  __device__ int num_gemms() const { return 1 + p.n_steps * (p.L * 4 + 1); }
  __device__ Gemm gemm(int i) const {
    Gemm g;
    const int B = p.B;
    if (i == 0) {   // small_to_mtp projection of step 1 (2 rows per frame)
      g.w = p.w_proj; g.s = p.s_proj; g.n_mt = p.d / kTileM; g.Kdim = p.th; g.acc = p.xres; g.ld = p.d; g.R = 2 * B;
    } else {
      const int j = i - 1, per_step = p.L * 4 + 1, step = j / per_step + 1, r = j % per_step;
      const int R = step == 1 ? 2 * B : B;
      if (r == p.L * 4) {   // lm_head[step-1]
        g.w = p.w_head[step - 1]; g.s = p.s_head[step - 1]; g.n_mt = p.V / kTileM; g.Kdim = p.d;
        g.acc = p.logits; g.ld = p.V; g.R = B;
      } else {
        const PLayer& L = p.layer[r / 4];
        switch (r % 4) {
          case 0: g.w = L.w_qkv; g.s = L.s_qkv; g.n_mt = (p.qw + 2 * p.kvw) / kTileM; g.Kdim = p.d;
                  g.acc = p.acc_qkv; g.ld = p.qw + 2 * p.kvw; break;
          case 1: g.w = L.w_o; g.s = L.s_o; g.n_mt = p.d / kTileM; g.Kdim = p.qw; g.acc = p.xres; g.ld = p.d; break;
          case 2: g.w = L.w_gu; g.s = L.s_gu; g.n_mt = 2 * p.F / kTileM; g.Kdim = p.d; g.acc = p.acc_gu;
                  g.ld = 2 * p.F; break;
          default: g.w = L.w_d; g.s = L.s_d; g.n_mt = p.d / kTileM; g.Kdim = p.F; g.acc = p.xres; g.ld = p.d; break;
        }
        g.R = R;
      }
    }
    g.n_ks = g.Kdim / kKs;
    return g;
  }
};

// ---------------------------------------------------------------------------
// grid barrier (consumer threads only)
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool grid_barrier(const PParams& p, unsigned int target) {
  named_bar(BAR_ALL, kConsumers);
  __shared__ int s_abort;
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(p.bar, 1u);
    int ab = 0;
    if (ld_acquire_u32(p.bar) < target) {
      const long long t0 = clock64();
      while (ld_acquire_u32(p.bar) < target) {
        if (*(volatile int*)p.abort_flag) { ab = 1; break; }
        if (clock64() - t0 > kSpinLimit) {
          set_status(p.status, QP_ERR_TIMEOUT);
          atomicExch(p.abort_flag, 1);
          ab = 1;
          break;
        }
      }
    }
    __threadfence();
    s_abort = ab;
  }
  named_bar(BAR_ALL, kConsumers);
  return s_abort == 0;
}

__device__ __forceinline__ void abort_all(const PParams& p) {
  set_status(p.status, QP_ERR_TIMEOUT);
  atomicExch(p.abort_flag, 1);
}

// Sum over the 128 threads of one half (4 warps) of the consumers.
__device__ __forceinline__ float half_sum(float v, float* red4, int half) {
  const int lane = threadIdx.x & 31, w = (threadIdx.x >> 5) & 3;
  v = warp_sum(v);
  if (lane == 0) red4[w] = v;
  named_bar(BAR_H0 + half, 128);
  const float s = red4[0] + red4[1] + red4[2] + red4[3];
  named_bar(BAR_H0 + half, 128);
  return s;
}

// Sum / max over all 256 consumer threads.
__device__ __forceinline__ float all_sum(float v, Smem& sm) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  v = warp_sum(v);
  if (lane == 0) sm.red[0][w] = v;
  named_bar(BAR_ALL, kConsumers);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) s += sm.red[0][i];
  named_bar(BAR_ALL, kConsumers);
  return s;
}

// ---------------------------------------------------------------------------
// elementwise phases
// ---------------------------------------------------------------------------

// Step 1 inputs: act rows 2b = f16(H[b]) and 2b+1 = f16(E0[q0[b]]) in the
// projection's operand layout; residual rows start at the projection bias.
__device__ void phase_prep(const PParams& p) {
  const int R = 2 * p.B;
  const Chunking c = chunking(R);
  for (int r = blockIdx.x; r < R; r += gridDim.x) {
    const int b = r >> 1;
    int q = 0;
    if (r & 1) {
      q = p.q0[b];
      if (q < 0 || q >= p.q0_vocab) {
        if (threadIdx.x == 0) set_status(p.status, QP_ERR_BAD_TOKEN);
        q = q < 0 ? 0 : p.q0_vocab - 1;
      }
    }
    for (int k = threadIdx.x * 4; k < p.th; k += kConsumers * 4) {
      float v[4];
      if (r & 1) {
        const uint2 e = *reinterpret_cast<const uint2*>(p.e0 + size_t(q) * p.th + k);
        v[0] = bf16_bits_to_f32(e.x & 0xffff); v[1] = bf16_bits_to_f32(e.x >> 16);
        v[2] = bf16_bits_to_f32(e.y & 0xffff); v[3] = bf16_bits_to_f32(e.y >> 16);
      } else {
        const float4 h = *reinterpret_cast<const float4*>(p.H + size_t(b) * p.th + k);
        v[0] = h.x; v[1] = h.y; v[2] = h.z; v[3] = h.w;
      }
      uint2 o;
      o.x = uint32_t(f32_to_f16_bits(v[0])) | (uint32_t(f32_to_f16_bits(v[1])) << 16);
      o.y = uint32_t(f32_to_f16_bits(v[2])) | (uint32_t(f32_to_f16_bits(v[3])) << 16);
      *reinterpret_cast<uint2*>(p.act + act_off(r, k, p.th, c)) = o;
    }
    for (int k = threadIdx.x; k < p.d; k += kConsumers) p.xres[size_t(r) * p.d + k] = p.b_proj[k];
  }
}

// act = f16(RMSNorm(xres[src row]) * w) in the layout for R rows; zero the
// next GEMM's accumulator rows.
__device__ void phase_norm(const PParams& p, Smem& sm, int R, int src_stride, int src_off, const float* w,
                           float* zero_acc, int zero_ld) {
  const Chunking c = chunking(R);
  for (int r = blockIdx.x; r < R; r += gridDim.x) {
    const float* x = p.xres + (size_t(r) * src_stride + src_off) * p.d;
    float v[4][4];
    float ss = 0.f;
    int n = 0;
    for (int k = threadIdx.x * 4; k < p.d; k += kConsumers * 4, ++n) {
      const float4 t = __ldcg(reinterpret_cast<const float4*>(x + k));
      v[n][0] = t.x; v[n][1] = t.y; v[n][2] = t.z; v[n][3] = t.w;
      ss += t.x * t.x + t.y * t.y + t.z * t.z + t.w * t.w;
    }
    ss = all_sum(ss, sm);
    const float inv = rsqrtf(ss / float(p.d) + p.eps);
    n = 0;
    for (int k = threadIdx.x * 4; k < p.d; k += kConsumers * 4, ++n) {
      uint2 o;
      o.x = uint32_t(f32_to_f16_bits(v[n][0] * inv * w[k])) | (uint32_t(f32_to_f16_bits(v[n][1] * inv * w[k + 1])) << 16);
      o.y = uint32_t(f32_to_f16_bits(v[n][2] * inv * w[k + 2])) | (uint32_t(f32_to_f16_bits(v[n][3] * inv * w[k + 3])) << 16);
      *reinterpret_cast<uint2*>(p.act + act_off(r, k, p.d, c)) = o;
    }
    if (zero_acc)
      for (int k = threadIdx.x * 4; k < zero_ld; k += kConsumers * 4)
        *reinterpret_cast<float4*>(zero_acc + size_t(r) * zero_ld + k) = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// Per-head RMSNorm then rotate-half RoPE of a 128-vector held one element
// per thread of a half.
__device__ __forceinline__ float head_norm_rope(float v, const float* nw, float eps, const float2* cs_row,
                                                Smem& sm, int half) {
  const int t = threadIdx.x & 127;
  const float ss = half_sum(v * v, sm.red[half], half);
  const float n = v * rsqrtf(ss / 128.f + eps) * nw[t];
  sm.xs[half][t] = n;
  named_bar(BAR_H0 + half, 128);
  const float2 cs = cs_row[t & 63];
  const float r = t < 64 ? n * cs.x - sm.xs[half][t + 64] * cs.y : n * cs.x + sm.xs[half][t - 64] * cs.y;
  named_bar(BAR_H0 + half, 128);
  return r;
}

// Attention of one (frame, kv head): per-head norms and RoPE of the new
// position(s), KV cache append, causal softmax over positions 0..pos for
// every q head of the group; output into the O-proj operand.
__device__ void phase_attn(const PParams& p, Smem& sm, int l, int P, int pos0) {
  const int B = p.B, R = B * P, ctx = p.n_steps + 1, grp = p.n_q / p.n_kv;
  const int qkvw = p.qw + 2 * p.kvw;
  const Chunking c = chunking(R);
  const int half = threadIdx.x >> 7, t = threadIdx.x & 127, lane = threadIdx.x & 31, wq = (threadIdx.x >> 5) & 3;
  const PLayer& L = p.layer[l];
  float* kv_l = p.kv + size_t(l) * p.Bmax * ctx * 2 * p.kvw;
  for (int item = blockIdx.x; item < B * p.n_kv; item += gridDim.x) {
    const int b = item / p.n_kv, j = item % p.n_kv;
    float* kvb = kv_l + size_t(b) * ctx * 2 * p.kvw;
    for (int pp = 0; pp < P; ++pp) {
      const int r = b * P + pp, pos = pos0 + pp;
      if (half == 0) {
        const float kr = __ldcg(p.acc_qkv + size_t(r) * qkvw + p.qw + j * 128 + t);
        const float ko = head_norm_rope(kr, L.k_norm, p.eps, p.rope_cs + pos * 64, sm, 0);
        kvb[(size_t(pos) * 2 + 0) * p.kvw + j * 128 + t] = ko;
      } else {
        kvb[(size_t(pos) * 2 + 1) * p.kvw + j * 128 + t] =
            __ldcg(p.acc_qkv + size_t(r) * qkvw + p.qw + p.kvw + j * 128 + t);
      }
    }
    named_bar(BAR_ALL, kConsumers);
    const float scale = rsqrtf(128.f);
    for (int pp = 0; pp < P; ++pp) {
      const int r = b * P + pp, pos = pos0 + pp;
      for (int gi = half; gi < grp; gi += 2) {
        const int hq = j * grp + gi;
        const float qr = __ldcg(p.acc_qkv + size_t(r) * qkvw + hq * 128 + t);
        const float qo = head_norm_rope(qr, L.q_norm, p.eps, p.rope_cs + pos * 64, sm, half);
        sm.xs[half][t] = qo;
        named_bar(BAR_H0 + half, 128);
        for (int i = wq; i <= pos; i += 4) {
          const float* kr = kvb + (size_t(i) * 2 + 0) * p.kvw + j * 128;
          const float4 kk = __ldcg(reinterpret_cast<const float4*>(kr + lane * 4));
          float s = sm.xs[half][lane * 4] * kk.x + sm.xs[half][lane * 4 + 1] * kk.y +
                    sm.xs[half][lane * 4 + 2] * kk.z + sm.xs[half][lane * 4 + 3] * kk.w;
          s = warp_sum(s);
          if (lane == 0) sm.sc[half][i] = s * scale;
        }
        named_bar(BAR_H0 + half, 128);
        float mx = -INFINITY;
        for (int i = 0; i <= pos; ++i) mx = fmaxf(mx, sm.sc[half][i]);
        float den = 0.f, o = 0.f;
        for (int i = 0; i <= pos; ++i) {
          const float e = expf(sm.sc[half][i] - mx);
          den += e;
          o += e * __ldcg(kvb + (size_t(i) * 2 + 1) * p.kvw + j * 128 + t);
        }
        p.act[act_off(r, hq * 128 + t, p.qw, c)] = f32_to_f16_bits(o / den);
        named_bar(BAR_H0 + half, 128);
      }
    }
    named_bar(BAR_ALL, kConsumers);
  }
}

// act = f16(silu(gate) * up) for R rows.
__device__ void phase_swiglu(const PParams& p, int R) {
  const Chunking c = chunking(R);
  const int F = p.F;
  for (int r = blockIdx.x; r < R; r += gridDim.x) {
    const float* gu = p.acc_gu + size_t(r) * 2 * F;
    for (int k = threadIdx.x * 4; k < F; k += kConsumers * 4) {
      const float4 g = __ldcg(reinterpret_cast<const float4*>(gu + k));
      const float4 u = __ldcg(reinterpret_cast<const float4*>(gu + F + k));
      uint2 o;
      o.x = uint32_t(f32_to_f16_bits(silu_f(g.x) * u.x)) | (uint32_t(f32_to_f16_bits(silu_f(g.y) * u.y)) << 16);
      o.y = uint32_t(f32_to_f16_bits(silu_f(g.z) * u.z)) | (uint32_t(f32_to_f16_bits(silu_f(g.w) * u.w)) << 16);
      *reinterpret_cast<uint2*>(p.act + act_off(r, k, F, c)) = o;
    }
  }
}

// Decision of step `step` for each frame: greedy argmax, or Gumbel-max over
// the top-k of logits / T.  Writes the code, the logits if asked, and the
// next position's residual row E[step-1][code].
__device__ void phase_decide(const PParams& p, Smem& sm, int step) {
  const int V = p.V, t = threadIdx.x, lane = t & 31, w = t >> 5;
  for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
    const float* l = p.logits + size_t(b) * V;
    if (p.out_logits) {
      float* o = p.out_logits + (size_t(b) * p.n_steps + (step - 1)) * V;
      for (int i = t; i < V; i += kConsumers) o[i] = __ldcg(l + i);
    }
    unsigned long long best = 0ull;
    if (p.temperature <= 0.f) {
      for (int i = t; i < V; i += kConsumers) {
        const unsigned long long pk = pack_argmax(__ldcg(l + i), i);
        best = pk > best ? pk : best;
      }
    } else {
      const float T = p.temperature;
      for (int i = t; i < V; i += kConsumers) sm.keys[i] = f32_order_key(__ldcg(l + i) / T);
      uint32_t prefix = 0, mask = 0;
      int remaining = p.top_k;
      for (int shift = 24; shift >= 0; shift -= 8) {
        sm.hist[t] = 0;
        named_bar(BAR_ALL, kConsumers);
        for (int i = t; i < V; i += kConsumers) {
          const uint32_t k = sm.keys[i];
          if ((k & mask) == prefix) atomicAdd(&sm.hist[(k >> shift) & 255], 1);
        }
        named_bar(BAR_ALL, kConsumers);
        if (t == 0) {
          int cum = 0, sel = 0;
          for (int dg = 255; dg >= 0; --dg) {
            if (cum + sm.hist[dg] >= remaining) { sel = dg; break; }
            cum += sm.hist[dg];
          }
          sm.sh_int[0] = sel;
          sm.sh_int[1] = remaining - cum;
        }
        named_bar(BAR_ALL, kConsumers);
        prefix |= uint32_t(sm.sh_int[0]) << shift;
        mask |= 255u << shift;
        remaining = sm.sh_int[1];
        named_bar(BAR_ALL, kConsumers);
      }
      const uint32_t kth = prefix;
      const int per = (V + kConsumers - 1) / kConsumers;
      const int lo = t * per, hi = min(V, lo + per);
      int cnt = 0;
      for (int i = lo; i < hi; ++i) cnt += sm.keys[i] == kth;
      sm.chunk_cnt[t] = cnt;
      named_bar(BAR_ALL, kConsumers);
      if (t == 0) {
        int run = 0;
        for (int i = 0; i < kConsumers; ++i) { const int cc = sm.chunk_cnt[i]; sm.chunk_cnt[i] = run; run += cc; }
      }
      named_bar(BAR_ALL, kConsumers);
      int eq_rank = sm.chunk_cnt[t];
      const float* gb = p.gumbel + (size_t(b) * p.n_steps + (step - 1)) * V;
      for (int i = lo; i < hi; ++i) {
        const uint32_t k = sm.keys[i];
        bool in = k > kth;
        if (k == kth) { in = eq_rank < remaining; ++eq_rank; }
        if (in) {
          const float z = __ldcg(l + i) / T;
          const unsigned long long pk = pack_argmax(z + gb[i], i);
          best = pk > best ? pk : best;
        }
      }
    }
    best = warp_max_u64(best);
    if (lane == 0) sm.redu[w] = best;
    named_bar(BAR_ALL, kConsumers);
    if (t == 0) {
      unsigned long long v = sm.redu[0];
      for (int i = 1; i < 8; ++i) v = sm.redu[i] > v ? sm.redu[i] : v;
      const int code = unpack_argmax_index(v);
      p.out_codes[size_t(b) * p.n_steps + (step - 1)] = code;
      int nc = p.forced ? p.forced[size_t(b) * p.n_steps + (step - 1)] : code;
      if (nc < 0 || nc >= V) {
        set_status(p.status, QP_ERR_BAD_TOKEN);
        nc = nc < 0 ? 0 : V - 1;
      }
      sm.sh_int[2] = nc;
    }
    named_bar(BAR_ALL, kConsumers);
    if (step < p.n_steps) {
      const uint16_t* e = p.embed[step - 1] + size_t(sm.sh_int[2]) * p.d;
      for (int i = t; i < p.d; i += kConsumers) p.xres[size_t(b) * p.d + i] = bf16_bits_to_f32(e[i]);
    }
    named_bar(BAR_ALL, kConsumers);
  }
}

// ---------------------------------------------------------------------------
// GEMM phase, consumer side
// ---------------------------------------------------------------------------
__device__ bool phase_gemm(const PParams& p, Smem& sm, const Gemm& g, int gemm_idx, uint32_t& slot_it,
                           uint32_t& act_it, uint32_t& mma_it) {
  const Chunking c = chunking(g.R);
  const int total = c.n_chunks * g.n_mt * g.n_ks;
  int beg, end;
  my_slices(total, gemm_idx, beg, end);
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t idesc = idesc_f16(kTileM, c.Nc);
  const uint32_t act_bytes = uint32_t(kKs) * c.Nc * 2;
  int* failed = &sm.sh_int[3];   // a wait ran out: unwind the whole grid
  if (t == 0) {
    *failed = 0;
    if (beg < end) fence_proxy_async_global();
  }
  named_bar(BAR_ALL, kConsumers);
  for (int s = beg; s < end; ++s) {
    const int ks = s % g.n_ks, tt = s / g.n_ks, mt = tt % g.n_mt, ch = tt / g.n_mt;
    const bool first = (s == beg) || ks == 0;
    const bool last = (s == end - 1) || ks == g.n_ks - 1;
    const uint32_t slot = slot_it % kNSlot, spar = (slot_it / kNSlot) & 1;
    ++slot_it;
    if (t == 0) {
      const uint16_t* src = p.act + size_t(ch) * g.Kdim * c.Nc + size_t(ks) * kKs * c.Nc;
      mbar_expect_tx(&sm.actbar, act_bytes);
      bulk_g2s(sm.actb, src, act_bytes, &sm.actbar);
    }
    const uint8_t* a_src = sm.slot[slot];
    if (p.q8) {
      if (!mbar_wait(&sm.full[slot], spar)) atomicOr(failed, 1);
      // dequantise the int8 slice into the f16 operand buffer (same order)
      const int8_t* qv = reinterpret_cast<const int8_t*>(sm.slot[slot]);
      const __half* sc = reinterpret_cast<const __half*>(sm.slot[slot] + kQ8Bytes);
      uint16_t* dq = reinterpret_cast<uint16_t*>(sm.deq);
      for (int e = t * 16; e < kTileM * kKs; e += kConsumers * 16) {
        // e indexes [k8][m8][8 rows][8 k]; 16 values = 2 rows of one core matrix
        const int4 raw = *reinterpret_cast<const int4*>(qv + e);
        const int8_t* q = reinterpret_cast<const int8_t*>(&raw);
        uint32_t out[8];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int ee = e + h2 * 8;
          const int k8 = ee >> 10, m = ((ee >> 6) & 15) * 8 + ((ee >> 3) & 7);
          const float dsc = __half2float(sc[(k8 >> 2) * kTileM + m]);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            out[h2 * 4 + i] = uint32_t(f32_to_f16_bits(q8_0_operand(dsc, q[h2 * 8 + 2 * i]))) |
                              (uint32_t(f32_to_f16_bits(q8_0_operand(dsc, q[h2 * 8 + 2 * i + 1]))) << 16);
        }
        *reinterpret_cast<uint4*>(dq + e) = make_uint4(out[0], out[1], out[2], out[3]);
        *reinterpret_cast<uint4*>(dq + e + 8) = make_uint4(out[4], out[5], out[6], out[7]);
      }
      fence_proxy_async_shared();
      named_bar(BAR_ALL, kConsumers);
      if (t == 0) mbar_arrive(&sm.empty[slot]);
      a_src = sm.deq;
    }
    if (t == 0) {
      if (!p.q8 && !mbar_wait(&sm.full[slot], spar)) *failed = 1;
      if (!mbar_wait(&sm.actbar, act_it & 1)) *failed = 1;
    }
    if (t == 0 && !*failed) {
      tc_fence_after();
      const uint32_t a0 = smem_u32(a_src), b0 = smem_u32(sm.actb);
#pragma unroll
      for (int j = 0; j < kKs / 16; ++j) {
        const uint64_t ad = smem_desc(a0 + j * 2 * (kTileM / 8) * 128, (kTileM / 8) * 128, 128);
        const uint64_t bd = smem_desc(b0 + j * 2 * (c.Nc / 8) * 128, (c.Nc / 8) * 128, 128);
        mma_f16(sm.tmem_base, ad, bd, idesc, (first && j == 0) ? 0u : 1u);
      }
      if (!p.q8) mma_commit(&sm.empty[slot]);
      mma_commit(&sm.mmabar);
      if (!mbar_wait(&sm.mmabar, mma_it & 1)) *failed = 1;
      tc_fence_before();
    }
    ++act_it;
    ++mma_it;
    named_bar(BAR_ALL, kConsumers);
    if (*failed) {
      if (t == 0) {
        abort_all(p);
        mbar_wait(&sm.actbar, (act_it - 1) & 1);   // the operand copy may still be landing
      }
      return false;
    }
    if (last) {
      tc_fence_after();
      const int quarter = warp & 3, halfc = warp >> 2;
      const int m = mt * kTileM + quarter * 32 + lane;
      const int cols = c.Nc / 2;
      for (int col = halfc * cols; col < (halfc + 1) * cols; col += 8) {
        float v[8];
        tmem_ld8(sm.tmem_base + (uint32_t(quarter * 32) << 16) + uint32_t(col), v);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int n = ch * c.Nc + col + i;
          if (n < g.R) red_add_f32(g.acc + size_t(n) * g.ld + m, v[i]);
        }
      }
      tc_fence_before();
      named_bar(BAR_ALL, kConsumers);
    }
  }
  return true;
}

// ---------------------------------------------------------------------------
// producer warp: stream this CTA's weight slices for every GEMM phase
// ---------------------------------------------------------------------------
__device__ void producer(const PParams& p, Smem& sm) {
  const Prog prog(p);
  const int ng = prog.num_gemms();
  const uint64_t pol = policy_evict_first();
  uint32_t it = 0;
  for (int gi = 0; gi < ng; ++gi) {
    const Gemm g = prog.gemm(gi);
    const Chunking c = chunking(g.R);
    const int total = c.n_chunks * g.n_mt * g.n_ks;
    int beg, end;
    my_slices(total, gi, beg, end);
    for (int s = beg; s < end; ++s) {
      const int ks = s % g.n_ks, mt = (s / g.n_ks) % g.n_mt;
      const uint32_t slot = it % kNSlot, u = it / kNSlot;
      if (u > 0) {
        bool done = false;
        const long long t0 = clock64();
        while (!(done = mbar_try_wait(&sm.empty[slot], (u - 1) & 1))) {
          if (*(volatile int*)p.abort_flag || clock64() - t0 > kSpinLimit) break;
        }
        if (!done) {
          abort_all(p);
          // drain copies still in flight into this CTA's shared memory
          for (uint32_t k = (it >= kNSlot ? it - kNSlot : 0); k < it; ++k)
            mbar_wait(&sm.full[k % kNSlot], (k / kNSlot) & 1);
          return;
        }
      }
      const size_t tile = size_t(mt) * g.n_ks + ks;
      if (p.q8) {
        mbar_expect_tx(&sm.full[slot], kQ8Bytes + kQ8ScaleBytes);
        bulk_g2s_stream(sm.slot[slot], g.w + tile * kQ8Bytes, kQ8Bytes, &sm.full[slot], pol);
        bulk_g2s_stream(sm.slot[slot] + kQ8Bytes, reinterpret_cast<const uint8_t*>(g.s) + tile * kQ8ScaleBytes,
                        kQ8ScaleBytes, &sm.full[slot], pol);
      } else {
        mbar_expect_tx(&sm.full[slot], kSlotBytes);
        bulk_g2s_stream(sm.slot[slot], g.w + tile * kSlotBytes, kSlotBytes, &sm.full[slot], pol);
      }
      ++it;
    }
  }
  // every slot the consumers did not take (abort path) must land before exit
  for (uint32_t k = (it >= kNSlot ? it - kNSlot : 0); k < it; ++k) mbar_wait(&sm.full[k % kNSlot], (k / kNSlot) & 1);
}

__global__ void __launch_bounds__(kThreads, 1) k_frames(const PParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int t = threadIdx.x, warp = t >> 5;
  if (t == 0) {
    for (int i = 0; i < kNSlot; ++i) { mbar_init(&sm.full[i], 1); mbar_init(&sm.empty[i], 1); }
    mbar_init(&sm.actbar, 1);
    mbar_init(&sm.mmabar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(&sm.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == kConsumers / 32) {
    if ((t & 31) == 0) producer(p, sm);
    return;
  }

  const Prog prog(p);
  uint32_t slot_it = 0, act_it = 0, mma_it = 0, phase = 0;
  int gemm_idx = 0;
  const unsigned G = gridDim.x;
  bool alive = true;
  auto barrier = [&]() {
    ++phase;
    alive = grid_barrier(p, phase * G);
    return alive;
  };
  auto gemm = [&]() {
    phase_gemm(p, sm, prog.gemm(gemm_idx), gemm_idx, slot_it, act_it, mma_it);
    ++gemm_idx;
    return barrier();
  };
  const int B = p.B, qkvw = p.qw + 2 * p.kvw;

  do {
    phase_prep(p);
    if (!barrier()) break;
    if (!gemm()) break;   // projection into xres
    for (int step = 1; step <= p.n_steps && alive; ++step) {
      const int P = step == 1 ? 2 : 1, R = B * P, pos0 = step == 1 ? 0 : step;
      for (int l = 0; l < p.L && alive; ++l) {
        const PLayer& L = p.layer[l];
        phase_norm(p, sm, R, 1, 0, L.attn_norm, p.acc_qkv, qkvw);
        if (!barrier()) break;
        if (!gemm()) break;                 // QKV
        phase_attn(p, sm, l, P, pos0);
        if (!barrier()) break;
        if (!gemm()) break;                 // O-proj into xres
        phase_norm(p, sm, R, 1, 0, L.ffn_norm, p.acc_gu, 2 * p.F);
        if (!barrier()) break;
        if (!gemm()) break;                 // gate/up
        phase_swiglu(p, R);
        if (!barrier()) break;
        if (!gemm()) break;                 // down into xres
      }
      if (!alive) break;
      phase_norm(p, sm, B, P, P - 1, p.out_norm, p.logits, p.V);
      if (!barrier()) break;
      if (!gemm()) break;                   // lm_head
      phase_decide(p, sm, step);
      if (!barrier()) break;
    }
  } while (false);

  // all tcgen05 work of this CTA is complete (every MMA was waited on)
  tc_fence_before();
  named_bar(BAR_ALL, kConsumers);
  tc_fence_after();
  if (warp == 0) tmem_dealloc(sm.tmem_base, kTmemCols);
}

// ---------------------------------------------------------------------------
// weight packing (load time)
// ---------------------------------------------------------------------------

// bf16 row-major [N, K] -> f16 packed tiles [N/128][K/8][16][8][8].
__global__ void k_pack_f16(const uint16_t* __restrict__ src, int N, int K, uint16_t* __restrict__ dst) {
  const size_t total = size_t(N) * (K / 8);
  for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < total; i += size_t(gridDim.x) * blockDim.x) {
    const int n = int(i / (K / 8)), k8 = int(i % (K / 8));
    const int mt = n / kTileM, r = n % kTileM;
    const uint4 v = *reinterpret_cast<const uint4*>(src + size_t(n) * K + k8 * 8);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = bf16_bits_to_f32(w[j] & 0xffff), hi = bf16_bits_to_f32(w[j] >> 16);
      o[j] = uint32_t(f32_to_f16_bits(lo)) | (uint32_t(f32_to_f16_bits(hi)) << 16);
    }
    const size_t off = size_t(mt) * K * kTileM + size_t(k8) * (kTileM * 8) + (r >> 3) * 64 + (r & 7) * 8;
    *reinterpret_cast<uint4*>(dst + off) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Q8_0 (int8 [N, K] + f16 scales [N, K/32]) -> packed int8 tiles in the same
// element order, and scales [N/128][K/128][4][128].
__global__ void k_pack_q8(const int8_t* __restrict__ qs, const __half* __restrict__ d, int N, int K,
                          int8_t* __restrict__ dq, __half* __restrict__ ds) {
  const size_t total = size_t(N) * (K / 8);
  for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < total; i += size_t(gridDim.x) * blockDim.x) {
    const int n = int(i / (K / 8)), k8 = int(i % (K / 8));
    const int mt = n / kTileM, r = n % kTileM;
    const uint2 v = *reinterpret_cast<const uint2*>(qs + size_t(n) * K + k8 * 8);
    const size_t off = size_t(mt) * K * kTileM + size_t(k8) * (kTileM * 8) + (r >> 3) * 64 + (r & 7) * 8;
    *reinterpret_cast<uint2*>(dq + off) = v;
    if ((k8 & 3) == 0) {
      const int k = k8 * 8, ks = k / kKs, kb = (k % kKs) / 32;
      ds[(size_t(mt) * (K / kKs) + ks) * (kKs / 32) * kTileM + kb * kTileM + r] = d[size_t(n) * (K / 32) + k / 32];
    }
  }
}

}  // namespace

size_t packed_bytes(int fmt, int N, int K) {
  if (fmt == WF_BF16) return size_t(N) * K * 2;
  return size_t(N) * K + size_t(N) * (K / 32) * 2;
}

cudaError_t pack_matrix(const QMat& src, PackedMat& dst, cudaStream_t s) {
  const size_t total = size_t(src.N) * (src.K / 8);
  const int grid = int(total / 256 + 1 < 8192 ? total / 256 + 1 : 8192);
  if (src.fmt == WF_BF16) {
    k_pack_f16<<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(src.w), src.N, src.K,
                                    reinterpret_cast<uint16_t*>(dst.w));
  } else {
    k_pack_q8<<<grid, 256, 0, s>>>(static_cast<const int8_t*>(src.w), src.scale, src.N, src.K,
                                   reinterpret_cast<int8_t*>(dst.w), dst.scale);
  }
  return cudaGetLastError();
}

size_t persistent_smem_bytes() { return sizeof(Smem) + 1024; }

qp_status run_frames_persistent(qp_handle* h, const RunArgs& a, cudaStream_t s) {
  const qp_geometry& g = h->g;
  if (a.temperature > 0.f && g.vocab > 8192) return QP_ERR_ARG;
  PParams p{};
  p.d = g.hidden; p.qw = g.n_q_heads * 128; p.kvw = g.n_kv_heads * 128; p.F = g.ffn; p.V = g.vocab;
  p.th = g.talker_hidden; p.L = g.layers; p.n_q = g.n_q_heads; p.n_kv = g.n_kv_heads; p.n_steps = g.n_steps;
  p.q0_vocab = g.q0_vocab; p.eps = g.rms_eps; p.q8 = h->wfmt == WF_Q8_0;
  p.w_proj = h->pproj.w; p.s_proj = h->pproj.scale; p.b_proj = h->b_proj; p.e0 = h->e0;
  for (int l = 0; l < g.layers; ++l) {
    const LayerW& L = h->layer[l];
    const PackedLayer& PL = h->player[l];
    p.layer[l] = {PL.qkv.w, PL.qkv.scale, PL.o.w, PL.o.scale, PL.gu.w, PL.gu.scale, PL.down.w, PL.down.scale,
                  L.attn_norm, L.q_norm, L.k_norm, L.ffn_norm};
  }
  p.out_norm = h->out_norm;
  for (int j = 0; j < g.n_steps; ++j) {
    p.embed[j] = h->embed[j];
    p.w_head[j] = h->phead[j].w;
    p.s_head[j] = h->phead[j].scale;
  }
  p.rope_cs = h->rope_cs;
  p.xres = h->X; p.act = h->pact; p.acc_qkv = h->qkv; p.acc_gu = h->gu; p.logits = h->logits; p.kv = h->kv;
  p.bar = h->sync_words; p.abort_flag = reinterpret_cast<int*>(h->sync_words + 1); p.status = h->status;
  p.Bmax = h->max_batch;
  p.B = a.B; p.H = a.H; p.q0 = a.q0; p.out_codes = a.out_codes; p.out_logits = a.out_logits; p.forced = a.forced;
  p.temperature = a.temperature; p.top_k = a.top_k; p.gumbel = a.gumbel;

  static bool attr_done[64] = {};
  const size_t smem = persistent_smem_bytes();
  if (h->device < 64 && !attr_done[h->device]) {
    if (cudaFuncSetAttribute(k_frames, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
      return QP_ERR_CUDA;
    attr_done[h->device] = true;
  }
  if (cudaMemsetAsync(h->sync_words, 0, 2 * sizeof(unsigned int), s) != cudaSuccess) return QP_ERR_CUDA;
  void* args[] = {&p};
  if (cudaLaunchCooperativeKernel(reinterpret_cast<void*>(k_frames), dim3(h->num_sms), dim3(kThreads), args, smem,
                                  s) != cudaSuccess) {
    cudaGetLastError();
    return QP_ERR_CUDA;
  }
  return QP_OK;
}


// ---------------------------------------------------------------------------
// Allocation-free entry point.
//
// Callers whose device memory is owned by someone else cannot have this
// library call cudaMalloc on their behalf: a process whose framework
// allocator has already reserved the GPU's memory, or a real-time audio path
// that forbids allocation once it is running.  qp_predict_frames_static
// runs the same persistent kernel as qp_predict_frames, but its scratch (the
// residual stream, MMA operand, accumulators, logits, KV cache and barrier
// words) lives in the file-scope array below, which the CUDA runtime places
// in device memory when the library's module loads on a device, and which
// every device that loads the library holds until the process exits.  The
// weights still come from a handle the caller loaded beforehand.
// ---------------------------------------------------------------------------

constexpr size_t kStaticScratchBytes = size_t(8) << 20;   // 8 MiB per device
constexpr int kStaticMaxFrames = 8;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
void* g_static_ptr[kMaxDevices] = {};
bool g_static_attr[kMaxDevices] = {};

size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

// Byte layout of the scratch for B frames; returns the total.
struct StaticLayout {
  size_t xres, act, qkv, gu, logits, kv, sync, total;
};
StaticLayout static_layout(const qp_geometry& g, int B) {
  const size_t R = size_t(2) * B;
  const size_t qw = size_t(g.n_q_heads) * 128, kvw = size_t(g.n_kv_heads) * 128;
  size_t aw = g.hidden;
  if (qw > aw) aw = qw;
  if (size_t(g.ffn) > aw) aw = g.ffn;
  if (size_t(g.talker_hidden) > aw) aw = g.talker_hidden;
  const size_t r16 = (R + 15) / 16 * 16;
  const size_t act_rows = r16 <= size_t(kMaxNc) ? r16 : (R + kMaxNc - 1) / kMaxNc * kMaxNc;
  StaticLayout L{};
  size_t off = 0;
  L.xres = off;   off += align256(R * g.hidden * 4);
  L.act = off;    off += align256(act_rows * aw * 2);
  L.qkv = off;    off += align256(R * (qw + 2 * kvw) * 4);
  L.gu = off;     off += align256(R * 2 * size_t(g.ffn) * 4);
  L.logits = off; off += align256(size_t(B) * g.vocab * 4);
  L.kv = off;     off += align256(size_t(g.layers) * B * (g.n_steps + 1) * 2 * kvw * 4);
  L.sync = off;   off += 256;
  L.total = off;
  return L;
}

}  // namespace

qp_status run_frames_static(qp_handle* h, const RunArgs& a, cudaStream_t s) {
  const qp_geometry& g = h->g;
  if (a.B < 1 || a.B > kStaticMaxFrames) return QP_ERR_ARG;
  const StaticLayout SL = static_layout(g, a.B);
  if (SL.total > kStaticScratchBytes) return QP_ERR_ARG;
  if (h->device < 0 || h->device >= kMaxDevices) return QP_ERR_ARG;
  // once per device, with that device current: the array's device address
  if (!g_static_ptr[h->device]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return QP_ERR_CUDA;
    }
    g_static_ptr[h->device] = ptr;
  }
  if (!g_static_attr[h->device]) {
    if (cudaFuncSetAttribute(k_frames, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(persistent_smem_bytes())) != cudaSuccess) {
      cudaGetLastError();
      return QP_ERR_CUDA;
    }
    g_static_attr[h->device] = true;
  }
  unsigned char* base = static_cast<unsigned char*>(g_static_ptr[h->device]);
  PParams p{};
  p.d = g.hidden; p.qw = g.n_q_heads * 128; p.kvw = g.n_kv_heads * 128; p.F = g.ffn; p.V = g.vocab;
  p.th = g.talker_hidden; p.L = g.layers; p.n_q = g.n_q_heads; p.n_kv = g.n_kv_heads; p.n_steps = g.n_steps;
  p.q0_vocab = g.q0_vocab; p.eps = g.rms_eps; p.q8 = h->wfmt == WF_Q8_0;
  p.w_proj = h->pproj.w; p.s_proj = h->pproj.scale; p.b_proj = h->b_proj; p.e0 = h->e0;
  for (int l = 0; l < g.layers; ++l) {
    const LayerW& L = h->layer[l];
    const PackedLayer& PL = h->player[l];
    p.layer[l] = {PL.qkv.w, PL.qkv.scale, PL.o.w, PL.o.scale, PL.gu.w, PL.gu.scale, PL.down.w, PL.down.scale,
                  L.attn_norm, L.q_norm, L.k_norm, L.ffn_norm};
  }
  p.out_norm = h->out_norm;
  for (int j = 0; j < g.n_steps; ++j) {
    p.embed[j] = h->embed[j];
    p.w_head[j] = h->phead[j].w;
    p.s_head[j] = h->phead[j].scale;
  }
  p.rope_cs = h->rope_cs;
  p.xres = reinterpret_cast<float*>(base + SL.xres);
  p.act = reinterpret_cast<uint16_t*>(base + SL.act);
  p.acc_qkv = reinterpret_cast<float*>(base + SL.qkv);
  p.acc_gu = reinterpret_cast<float*>(base + SL.gu);
  p.logits = reinterpret_cast<float*>(base + SL.logits);
  p.kv = reinterpret_cast<float*>(base + SL.kv);
  p.bar = reinterpret_cast<unsigned int*>(base + SL.sync);
  p.abort_flag = reinterpret_cast<int*>(base + SL.sync + 4);
  p.status = h->status;
  p.Bmax = a.B;
  p.B = a.B; p.H = a.H; p.q0 = a.q0; p.out_codes = a.out_codes; p.out_logits = a.out_logits; p.forced = nullptr;
  p.temperature = 0.f; p.top_k = 0; p.gumbel = nullptr;
  // the barrier counter and abort flag must start at zero; every other
  // buffer is written before it is read within the call
  if (cudaMemsetAsync(base + SL.sync, 0, 8, s) != cudaSuccess) {
    cudaGetLastError();
    return QP_ERR_CUDA;
  }
  void* args[] = {&p};
  if (cudaLaunchCooperativeKernel(reinterpret_cast<void*>(k_frames), dim3(h->num_sms), dim3(kThreads), args,
                                  persistent_smem_bytes(), s) != cudaSuccess) {
    cudaGetLastError();
    return QP_ERR_CUDA;
  }
  return QP_OK;
}

}  // namespace qp
