// The Code Predictor frame loop as ONE persistent cooperative kernel,
// scheduled as a dataflow over tiles.
//
// For a batch of B frames the call runs the whole 15-step loop
// ("テキスト音声合成モデルを50ミリ秒未満で応答させる方法", "Qwen3-TTSの最適化方法"
// item 3: a fixed GPU program instead of a host-driven sequence, over a
// preallocated KV cache):
//   step 1: rows 2b = small_to_mtp(H_b), 2b+1 = small_to_mtp(E0[q0_b]);
//   step k >= 2: row b = E[k-2][q_{k-1}];
//   5 layers per step: RMSNorm -> QKV -> per-head QK-norm + RoPE -> causal
//   GQA attention -> O + residual -> RMSNorm -> gate/up -> SwiGLU -> down +
//   residual; then output RMSNorm, lm_head[k-1] and the decision.
//
// Every weight contraction runs on the tcgen05 tensor cores as
//   D[128 weight rows, Nc activation rows] += W[128, 128-K slice] * act^T
// with f16 operands and f32 accumulators in TMEM.  Weights arrive packed in
// the MMA's shared-memory image (qp_weights.cu), one bulk copy per slice.
//
// Roles inside each CTA (one CTA per SM, all co-resident):
//   producer warp  streams the CTA's weight slices for the whole call through
//                  a ring of shared-memory slots;
//   dequant warps  (Q8_0 only) turn int8 slices into f16 operand slots;
//   MMA warp       waits until a slice's activation operand is published,
//                  bulk-copies it, issues the MMAs into one of two TMEM
//                  accumulators and commits;
//   consumer warps drain accumulators into f32 buffers (red.add, so slices
//                  of one tile may come from several CTAs), and run the
//                  elementwise work.
// There are no grid-wide barriers.  Each output tile carries a counter; once
// it is complete, the CTAs that added into the tile finish it, each its share
// of the rows: an x tile becomes the next GEMM's operand f16(x * w_norm) plus
// partial sums of squares (the next GEMM scales its output by 1/rms), a
// gate/up tile pair becomes the down operand silu(g)*u, a logits tile feeds
// the greedy argmax.  Attention runs one warp per (frame, kv head) as soon as that
// head's q/k/v tiles are complete.  Consumers wait only on work earlier in
// the one program order every CTA follows, so the earliest pending item can
// always run: no deadlock.  Every wait is bounded; one that runs out latches
// QP_ERR_TIMEOUT and sets an abort flag that every other wait honours.
#include <atomic>

#include "qp_device.cuh"
#include "../../include/qp_debug.h"

namespace qp {

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kDeqWarp0 = 10;
constexpr int kDeqThreads = 4 * 32;
// This translation unit's kernel: k_frames for 16-bit weights (10 warps:
// consumers, producer, MMA), or, built from qp_persistent_q8.cu, k_frames_q8
// for Q8_0 matrices, whose 4 more warps dequantise.  Without them a thread
// may hold 168 registers instead of 128, and the 16-bit kernel does not
// spill.
#ifndef QP_TILE_Q8
#define QP_TILE_Q8 0
#endif
constexpr bool kTileQ8 = QP_TILE_Q8 != 0;
constexpr int kThreads = (kConsumerWarps + 2 + (kTileQ8 ? 4 : 0)) * 32;   // 320 or 448

constexpr uint32_t kSlotBytes = kTileM * kKs * 2;              // 32 KB f16 slice
constexpr uint32_t kQ8Bytes = kTileM * kKs;                    // 16 KB int8 slice
constexpr uint32_t kQ8ScaleBytes = (kKs / 32) * kTileM * 2;    // 1 KB of scales
constexpr uint32_t kQ8SlotBytes = kQ8Bytes + kQ8ScaleBytes;
// A dequantised Q8_0 slice is two f16 images, hi = f16(d*q) and lo =
// f16(d*q - hi), whose sum is d*q exactly (below); they take two
// consecutive places of a ring of kNDeq 32 KB places, a 16-bit head slice
// among Q8_0 matrices one.
constexpr int kNSlotF16 = 4, kNSlotQ8 = 2, kNDeq = 3, kNAct = 2;
constexpr uint32_t kActBytes = kKs * kMaxNc * 2;               // 32 KB operand slice
constexpr uint32_t kTmemCols = 256;                            // two 128-column accumulators

// shared memory map (offsets from a 1 KB aligned base).  The 16-bit kernel
// has no dequantised places; the Q8_0 kernel's raw ring is smaller than the
// 16-bit ring, and its activation slots sit after the dequantised places.
constexpr uint32_t kOffRing = 0;                               // f16 slots, or Q8_0 raw slots
constexpr uint32_t kOffDeq = 35840;                            // Q8_0: dequantised places
constexpr uint32_t kOffAct = kTileQ8 ? kOffDeq + kNDeq * kSlotBytes : kNSlotF16 * kSlotBytes;   // activation slots
constexpr uint32_t kOffKeys = kOffAct + kNAct * kActBytes;     // top-k keys
constexpr uint32_t kOffMisc = kOffKeys + kMaxVocab * 4;
static_assert(kNSlotQ8 * kQ8SlotBytes <= kOffDeq, "raw Q8_0 slots overlap the dequantised ones");
static_assert(kSlotBytes / 2 <= kQ8SlotBytes && kNSlotQ8 >= 2, "a 16-bit slice takes two raw slots");
static_assert(kNDeq >= 2, "a Q8_0 slice takes two dequantised places");
static_assert(kOffDeq % 1024 == 0 && kOffAct % 1024 == 0, "operand images start on 1 KB boundaries");
static_assert(kNSlotF16 * kSlotBytes <= kOffAct, "f16 slots overlap the operand slots");

enum { BAR_CONS = 1, BAR_DEQ = 2, BAR_HALF0 = 3 };   // BAR_HALF0 + h: consumer half h (4 warps)
enum { G_PROJ = 0, G_QKV, G_O, G_GU, G_DOWN, G_HEAD };

struct Misc {
  uint64_t wfull[kNSlotF16], wempty[kNSlotF16];
  uint64_t dfull[kNDeq], dempty[kNDeq];
  uint64_t afull[kNAct], aempty[kNAct];
  uint64_t accfull[2], accempty[2];
  uint64_t mmadone;
  uint32_t tmem_base;
  int flag[4];
  int fail;       // a consumer wait gave up: every consumer warp leaves at the next section end
  unsigned evc;   // next slot of this CTA's consumer event log (tracing only)
  int deq_ok;     // broadcast of the dequant leader's waits
  float red[8];
  unsigned long long redu[8];
  int sel[2];
  int hist[256];
  TopkScratch topk[2];   // sampling: one frame per consumer half
  int hflag[2];
  float inv[kMaxNc];
};

struct PLayer {
  const uint8_t* w[4];     // qkv, o, gu, down (packed)
  const __half* s[4];
  const float* attn_norm; const float* q_norm; const float* k_norm; const float* ffn_norm;
};

struct PParams {
  int d, qw, kvw, F, V, th, L, n_q, n_kv, n_steps, q0_vocab;
  float eps;
  int q8;        // projection and layer matrices are Q8_0
  int q8_head;   // lm-heads are Q8_0 (else 16-bit, served from the dequantised slots when q8)
  bool embed_f16;   // embedding tables are f16, else bf16
  int proj_in;   // code tables are Talker-wide: each step's input passes through small_to_mtp
  const uint8_t* w_proj; const __half* s_proj; const float* b_proj; const uint16_t* e0;
  PLayer layer[kMaxLayers];
  const float* out_norm;
  const uint16_t* embed[kMaxSteps]; const float* embed_ss[kMaxSteps];
  const uint8_t* w_head[kMaxSteps]; const __half* s_head[kMaxSteps];
  const float2* rope_cs;
  // scratch
  float* x1; float* xk; uint16_t* a1[5]; uint16_t* ak[4]; uint16_t* ahead;
  float* acc1_qkv; float* acck_qkv; float* acc1_gu; float* acck_gu; float* logits;
  uint16_t* kv;   // f16 [layer][frame][pos][k|v][kv_width]
  int Bmax;
  // per-call synchronisation (zeroed before the launch)
  unsigned* tile_cnt; unsigned* ready; unsigned* ss_cnt; float* ss; unsigned* head_done;
  int* rexp;   // [gemm][row]: range exponent e of the operand row (f16(v * 2^-e); 0 = unscaled)
  unsigned long long* codepk; unsigned* decided; int* abort_flag; int* status;
  long long spin_limit;   // clock64 ticks a wait may take before the call aborts
  int det;                // deterministic mode: no split K; squared norms summed in tile order
  float* ss_part;         // deterministic mode: [gemm][x tile][row] partial sums of squares
  int withhold;           // testing (qp_debug.h): GEMM whose first tile count CTA run 0 skips; -1 none
  int NCH, MT, KS, NGEMM;
  unsigned long long* trace; int trace_n;
  // the call
  int B; const float* H; const int32_t* q0; int32_t* out_codes; float* out_logits; const int32_t* forced;
  float temperature; int top_k; const float* gumbel;
};

// Q8_0 matrices: only the Q8_0 build of the kernel has the dequantising warps.
__device__ __forceinline__ bool tq8(const PParams& p) { return kTileQ8 && p.q8; }

// ------------------------------------------------------------ event log
// With tracing on, each CTA also keeps an event log after the section stamps:
// consumer events in [0, 8192), MMA-warp events in [8192, 16384) of its
// region; one word = (globaltimer ns mod 2^48) << 16 | code << 12 | gemm.
enum {
  EV_READY = 1, EV_LANDED, EV_COMMIT,            // MMA warp, per slice / segment
  EV_ACC = 4, EV_REDS, EV_COUNTED, EV_LASTDONE,   // consumer epilogue, per segment
  EV_ATT_READY = 8, EV_ATT_DONE,                  // attention warp, per item
  EV_WEIGHTS = 10,                                // MMA warp: the slice's weights are in shared memory
  EV_DEC_READY = 11, EV_DEC_DONE = 12             // sampling: a frame's logits complete; its code published
};
__device__ __forceinline__ unsigned long long* ev_base(const PParams& p) {
  return p.trace ? p.trace + size_t(p.trace_n) * gridDim.x * 2 + size_t(blockIdx.x) * 16384 : nullptr;
}
__device__ __forceinline__ unsigned long long ev_word(int code, int gi) {
  return ((globaltimer_ns() & 0xFFFFFFFFFFFFull) << 16) | (unsigned long long)(code & 15) << 12 | unsigned(gi & 4095);
}
// Compiled in only with QP_TRACE (qp_debug.h): the hooks sit on the loop's
// critical path, where even untaken branches cost instruction fetch.
#ifdef QP_TRACE
__device__ __forceinline__ void ev_mma(const PParams& p, unsigned& idx, int code, int gi) {
  unsigned long long* b = ev_base(p);
  if (b && idx < 8192) b[8192 + idx++] = ev_word(code, gi);
}
__device__ __forceinline__ void ev_cons(const PParams& p, unsigned* evc, int code, int gi) {
  unsigned long long* b = ev_base(p);
  if (b) {
    const unsigned i = atomicAdd(evc, 1u);
    if (i < 8192) b[i] = ev_word(code, gi);
  }
}
#else
__device__ __forceinline__ void ev_mma(const PParams&, unsigned&, int, int) {}
__device__ __forceinline__ void ev_cons(const PParams&, unsigned*, int, int) {}
#endif

// ----------------------------------------------------------- the program
struct Ck { int Nc, n; };
__device__ __forceinline__ Ck chunking(int R) {
  const int r16 = (R + 15) & ~15;
  if (r16 <= kMaxNc) return {r16, 1};
  return {kMaxNc, (R + kMaxNc - 1) / kMaxNc};
}
__device__ __forceinline__ int rows_in(int R, Ck c, int ch) { return min(c.Nc, R - ch * c.Nc); }

// Element offset of (row n, feature k) in an operand buffer laid out
// [chunk][K/8][Nc/8][8 rows][8 k] for reduction length Kdim.
__device__ __forceinline__ size_t act_off(int n, int k, int Kdim, Ck c) {
  const int ch = n / c.Nc, nn = n - ch * c.Nc;
  return size_t(ch) * Kdim * c.Nc + (size_t((k >> 3) * (c.Nc >> 3) + (nn >> 3)) << 6) + ((nn & 7) << 3) + (k & 7);
}

struct GI {
  int kind, k, l, R, n_mt, n_ks, Kdim, ld;
  const uint8_t* w; const __half* s; const uint16_t* act; float* acc;
};

// The program: GEMM 0 is step 1's projection (rows H_b, E0[q0_b]); step k
// then has, with Talker-wide code tables and k >= 2, the projection of its
// input rows, then 4 GEMMs per layer (QKV, O, GU, down) and the head.
__device__ __forceinline__ int gi_base(const PParams& p, int k) {
  return 1 + (k - 1) * (4 * p.L + 1) + p.proj_in * (k - 1);
}
__device__ __forceinline__ int gi_of(const PParams& p, int k, int l, int t) { return gi_base(p, k) + 4 * l + t; }
__device__ __forceinline__ int gi_head(const PParams& p, int k) { return gi_base(p, k) + 4 * p.L; }
__device__ __forceinline__ int gi_proj(const PParams& p, int k) { return k == 1 ? 0 : gi_base(p, k) - 1; }

__device__ GI gemm_inst(const PParams& p, int gi) {
  GI g;
  const int B = p.B;
  int r = -1;   // the GEMM's place in its step: -1 the projection, 4L the head
  if (gi == 0) {
    g.k = 1;
  } else {
    const int per1 = 4 * p.L + 1, perk = per1 + p.proj_in;
    if (gi <= per1) {
      g.k = 1; r = gi - 1;
    } else {
      const int j = gi - 1 - per1;
      g.k = j / perk + 2; r = j % perk - p.proj_in;
    }
  }
  if (r < 0) {
    // step 1: rows H_b, E0[q0_b] into x1; step k >= 2: rows E[k-2][code_b] into xk
    g.kind = G_PROJ; g.l = 0; g.R = g.k == 1 ? 2 * B : B; g.n_mt = p.d / kTileM; g.Kdim = p.th;
    g.w = p.w_proj; g.s = p.s_proj; g.act = p.a1[0]; g.acc = g.k == 1 ? p.x1 : p.xk; g.ld = p.d;
  } else {
    const bool s1 = g.k == 1;
    if (r == 4 * p.L) {
      g.kind = G_HEAD; g.l = p.L - 1; g.R = B; g.n_mt = p.V / kTileM; g.Kdim = p.d;
      g.w = p.w_head[g.k - 1]; g.s = p.s_head[g.k - 1]; g.act = p.ahead; g.acc = p.logits; g.ld = p.V;
    } else {
      g.l = r / 4;
      g.R = s1 ? 2 * B : B;
      const PLayer& L = p.layer[g.l];
      const int t = r % 4;
      g.w = L.w[t]; g.s = L.s[t];
      switch (t) {
        case 0: g.kind = G_QKV; g.n_mt = (p.qw + 2 * p.kvw) / kTileM; g.Kdim = p.d;
                g.act = s1 ? p.a1[1] : p.ak[0]; g.acc = s1 ? p.acc1_qkv : p.acck_qkv; g.ld = p.qw + 2 * p.kvw; break;
        case 1: g.kind = G_O; g.n_mt = p.d / kTileM; g.Kdim = p.qw;
                g.act = s1 ? p.a1[2] : p.ak[1]; g.acc = s1 ? p.x1 : p.xk; g.ld = p.d; break;
        case 2: g.kind = G_GU; g.n_mt = 2 * p.F / kTileM; g.Kdim = p.d;
                g.act = s1 ? p.a1[3] : p.ak[2]; g.acc = s1 ? p.acc1_gu : p.acck_gu; g.ld = 2 * p.F; break;
        default: g.kind = G_DOWN; g.n_mt = p.d / kTileM; g.Kdim = p.F;
                 g.act = s1 ? p.a1[4] : p.ak[3]; g.acc = s1 ? p.x1 : p.xk; g.ld = p.d; break;
      }
    }
  }
  g.n_ks = g.Kdim / kKs;
  return g;
}

// This CTA's contiguous run [beg, end) of a GEMM's slices.  Slices are
// ordered (chunk, 128-row tile, K slice); runs rotate with the GEMM index.
// The GEMM's slices are ordered (chunk, 128-row tile, K slice) and cut into
// pieces: each tile's K range is split into S parts, S = the fewest that
// still gives every CTA a piece (1 once the tiles outnumber the CTAs), so a
// tile's partial sums pass through the f32 accumulator as few times as the
// grid allows.  This CTA takes a contiguous run of pieces -- a contiguous
// run [beg, end) of slices -- rotated with the GEMM index.
__device__ __forceinline__ int split_of(int tiles, int n_ks, int det) {
  return det ? 1 : max(1, min(n_ks, int(gridDim.x) / tiles));
}
__device__ __forceinline__ void my_run(int tiles, int n_ks, int gi, int& beg, int& end, int det) {
  const int G = gridDim.x, g = (blockIdx.x + gi * 37) % G;
  const int S = split_of(tiles, n_ks, det);
  const long long P = (long long)tiles * S;
  const int p0 = int(P * g / G), p1 = int(P * (g + 1) / G);
  beg = (p0 / S) * n_ks + ((p0 % S) * n_ks) / S;
  end = (p1 / S) * n_ks + ((p1 % S) * n_ks) / S;
}

// This CTA's place among the contributors of tile tt in my_run's split (the
// owners of the tile's S parts).  Returns the rank of this CTA (-1 if it
// holds no part of the tile) and sets n to the number of contributors.
// With fewer parts than CTAs each CTA holds at most one part, and the S
// owners need not be consecutive; otherwise every CTA holds a part and the
// owners are consecutive in the rotated CTA index.
__device__ __forceinline__ int tile_share(int tiles, int n_ks, int gi, int tt, int& n, int det) {
  const int G = gridDim.x, g = (blockIdx.x + gi * 37) % G;
  const int S = split_of(tiles, n_ks, det);
  const long long P = (long long)tiles * S, q0 = (long long)tt * S;
  if (P < G) {
    const long long p0 = P * g / G, p1 = P * (g + 1) / G;
    n = S;
    return p1 > p0 && p0 >= q0 && p0 < q0 + S ? int(p0 - q0) : -1;
  }
  // the owner of part q: the largest g with floor(P * g / G) <= q
  const int g0 = int(((q0 + 1) * G - 1) / P), g1 = int(((q0 + S) * G - 1) / P);
  n = g1 - g0 + 1;
  return g >= g0 && g <= g1 ? g - g0 : -1;
}

// sync-region accessors
__device__ __forceinline__ unsigned* tile_cnt(const PParams& p, int gi, int ch, int mt) {
  return p.tile_cnt + (size_t(gi) * p.NCH + ch) * p.MT + mt;
}
__device__ __forceinline__ unsigned* ready_cnt(const PParams& p, int gi, int ch, int ks) {
  return p.ready + (size_t(gi) * p.NCH + ch) * p.KS + ks;
}
__device__ __forceinline__ unsigned* ss_cnt(const PParams& p, int gi, int ch) { return p.ss_cnt + size_t(gi) * p.NCH + ch; }
__device__ __forceinline__ float* ss_at(const PParams& p, int gi, int row) { return p.ss + size_t(gi) * 2 * p.B + row; }
__device__ __forceinline__ int* rexp_at(const PParams& p, int gi, int row) { return p.rexp + size_t(gi) * 2 * p.B + row; }
// Deterministic mode: the partial sum of squares of x tile mt of a row.
__device__ __forceinline__ float* ss_part_at(const PParams& p, int gi, int mt, int row) {
  return p.ss_part + (size_t(gi) * (p.d / kTileM) + mt) * 2 * p.B + row;
}
// A row's sum of squares (complete): the accumulated word, or in
// deterministic mode the tiles' partial sums added in tile order.
__device__ __forceinline__ float ss_total(const PParams& p, int gi, int row) {
  if (!p.det) return __ldcg(ss_at(p, gi, row));
  float s = 0.f;
  for (int mt = 0; mt < p.d / kTileM; ++mt) s += __ldcg(ss_part_at(p, gi, mt, row));
  return s;
}
__device__ __forceinline__ unsigned* head_done(const PParams& p, int k, int ch) {
  return p.head_done + size_t(k - 1) * p.NCH + ch;
}

// ---------------------------------------------------------------- producer
// With Q8_0 matrices and 16-bit heads, a head slice (32 KB of f16) arrives
// as two 16 KB halves in two consecutive raw slots, and the dequantising
// warps copy it unchanged into the dequantised slot the MMA warp reads.
// Every slice thus takes the same path in program order: each mbarrier's
// waiters stay within one phase of it, which parity waits require.
__device__ __forceinline__ bool slice_is_q8(const PParams& p, const GI& G) {
  return tq8(p) && (G.kind != G_HEAD || p.q8_head);
}

__device__ void producer_role(const PParams& p, Misc& ms, uint8_t* smem) {
  const int nslot = tq8(p) ? kNSlotQ8 : kNSlotF16;
  const uint32_t stride = tq8(p) ? kQ8SlotBytes : kSlotBytes;
  const uint64_t pol = policy_evict_first();
  uint32_t it = 0;      // raw-slot copies issued
  for (int gi = 0; gi < p.NGEMM; ++gi) {
    const GI G = gemm_inst(p, gi);
    const Ck c = chunking(G.R);
    const bool q8g = slice_is_q8(p, G);
    int beg, end;
    my_run(c.n * G.n_mt, G.n_ks, gi, beg, end, p.det);
    for (int s = beg; s < end; ++s) {
      const int ks = s % G.n_ks, mt = (s / G.n_ks) % G.n_mt;
      if (tq8(p) && !q8g) {
        const size_t tile = size_t(mt) * G.n_ks + ks;
        for (int h = 0; h < 2; ++h, ++it) {
          const uint32_t slot = it % nslot, u = it / nslot;
          if (u > 0 && !mwait(p, &ms.wempty[slot], (u - 1) & 1)) goto drain;
          mbar_expect_tx(&ms.wfull[slot], kSlotBytes / 2);
          bulk_g2s_stream(smem + kOffRing + slot * stride, G.w + tile * kSlotBytes + h * (kSlotBytes / 2),
                          kSlotBytes / 2, &ms.wfull[slot], pol);
        }
        continue;
      }
      const uint32_t slot = it % nslot, u = it / nslot;
      if (u > 0 && !mwait(p, &ms.wempty[slot], (u - 1) & 1)) goto drain;
      {
        const size_t tile = size_t(mt) * G.n_ks + ks;
        uint8_t* dst = smem + kOffRing + slot * stride;
        if (tq8(p)) {
          mbar_expect_tx(&ms.wfull[slot], kQ8SlotBytes);
          bulk_g2s_stream(dst, G.w + tile * kQ8Bytes, kQ8Bytes, &ms.wfull[slot], pol);
          bulk_g2s_stream(dst + kQ8Bytes, reinterpret_cast<const uint8_t*>(G.s) + tile * kQ8ScaleBytes, kQ8ScaleBytes,
                          &ms.wfull[slot], pol);
        } else {
          mbar_expect_tx(&ms.wfull[slot], kSlotBytes);
          bulk_g2s_stream(dst, G.w + tile * kSlotBytes, kSlotBytes, &ms.wfull[slot], pol);
        }
      }
      ++it;
    }
  }
drain:
  // every copy issued into this CTA's shared memory lands before it exits
  for (uint32_t k = it > uint32_t(nslot) ? it - nslot : 0; k < it; ++k) mbar_wait(&ms.wfull[k % nslot], (k / nslot) & 1);
}

// --------------------------------------------------------- Q8_0 dequant
// Four int8 values (one 32-bit word, little-endian) times an f16 scale d, as
// two f16 quadruples hi and lo with hi + lo = d * q.  q is made exact in
// f16 as (1024 + (q + 128)) - 1152 -- the mantissa of an f16 in [1024, 2048)
// holds the integer; hi = d * q rounded once to the nearest f16 (one f16
// multiply), lo = d * q - hi from one fused multiply-add, rounded once.
// d * q - hi is a multiple of d's last place (q is an integer) and at most
// half of hi's, so it needs at most 7 significant bits and lo holds it
// exactly whenever d >= 2^-14 (the smallest normal f16): the pair is the
// stored weight d * q, with no rounding.
__device__ __forceinline__ void q8x4_to_f16x4_hilo(uint32_t w, __half2 d2, uint2& hi, uint2& lo) {
  const uint32_t u = w ^ 0x80808080u;                 // q + 128 in each byte
  const uint32_t b01 = __byte_perm(u, 0x64646464u, 0x5150);   // bytes 0,1 -> f16 0x64xx
  const uint32_t b23 = __byte_perm(u, 0x64646464u, 0x5352);   // bytes 2,3
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));   // 1152
  const __half2 qa = __hsub2(*reinterpret_cast<const __half2*>(&b01), bias);
  const __half2 qb = __hsub2(*reinterpret_cast<const __half2*>(&b23), bias);
  const __half2 ha = __hmul2(qa, d2), hb = __hmul2(qb, d2);
  const __half2 la = __hfma2(qa, d2, __hneg2(ha)), lb = __hfma2(qb, d2, __hneg2(hb));
  hi = make_uint2(*reinterpret_cast<const uint32_t*>(&ha), *reinterpret_cast<const uint32_t*>(&hb));
  lo = make_uint2(*reinterpret_cast<const uint32_t*>(&la), *reinterpret_cast<const uint32_t*>(&lb));
}

// Dequantised places: a ring of kNDeq 32 KB images that the dequantising
// warps fill in program order and the MMA warp empties in the same order;
// a Q8_0 slice takes two consecutive places (hi, lo), a 16-bit slice one.
__device__ void dequant_role(const PParams& p, Misc& ms, uint8_t* smem) {
  const int t = threadIdx.x - kDeqWarp0 * 32;
  uint32_t it = 0, rit = 0;   // dequantised places used; raw slots used
  for (int gi = 0; gi < p.NGEMM; ++gi) {
    const GI G = gemm_inst(p, gi);
    const Ck c = chunking(G.R);
    const bool q8g = slice_is_q8(p, G);
    int beg, end;
    my_run(c.n * G.n_mt, G.n_ks, gi, beg, end, p.det);
    for (int s = beg; s < end; ++s, it += q8g ? 2 : 1, rit += q8g ? 1 : 2) {
      const uint32_t rs = rit % kNSlotQ8, ru = rit / kNSlotQ8;
      const uint32_t rs2 = (rit + 1) % kNSlotQ8, ru2 = (rit + 1) / kNSlotQ8;
      const uint32_t ds = it % kNDeq, du = it / kNDeq, ds2 = (it + 1) % kNDeq, du2 = (it + 1) / kNDeq;
      if (t == 0) {   // the leader waits for every dequant thread, then broadcasts
        bool w = mwait(p, &ms.wfull[rs], ru & 1);
        if (w && !q8g) w = mwait(p, &ms.wfull[rs2], ru2 & 1);
        if (w && du > 0) w = mwait(p, &ms.dempty[ds], (du - 1) & 1);
        ms.deq_ok = w;
      }
      named_bar(BAR_DEQ, kDeqThreads);
      if (!ms.deq_ok) return;
      if (!q8g) {
        // a 16-bit slice: its two halves, unchanged
        uint4* dq4 = reinterpret_cast<uint4*>(smem + kOffDeq + ds * kSlotBytes);
        const uint4* h0 = reinterpret_cast<const uint4*>(smem + kOffRing + rs * kQ8SlotBytes);
        const uint4* h1 = reinterpret_cast<const uint4*>(smem + kOffRing + rs2 * kQ8SlotBytes);
        constexpr int kHalf4 = int(kSlotBytes / 2 / 16);
        for (int e = t; e < 2 * kHalf4; e += kDeqThreads) dq4[e] = e < kHalf4 ? h0[e] : h1[e - kHalf4];
        fence_proxy_async_shared();
        named_bar(BAR_DEQ, kDeqThreads);
        if (t == 0) {
          mbar_arrive(&ms.wempty[rs]);
          mbar_arrive(&ms.wempty[rs2]);
          mbar_arrive(&ms.dfull[ds]);
        }
        continue;
      }
      const uint8_t* src = smem + kOffRing + rs * kQ8SlotBytes;
      const int8_t* qv = reinterpret_cast<const int8_t*>(src);
      const __half* sc = reinterpret_cast<const __half*>(src + kQ8Bytes);
      // two passes, hi then lo, each published on its own: the MMA warp
      // multiplies the hi image while the lo image is written
      for (int pass = 0; pass < 2; ++pass) {
        if (pass == 1) {
          if (t == 0) ms.deq_ok = du2 == 0 || mwait(p, &ms.dempty[ds2], (du2 - 1) & 1);
          named_bar(BAR_DEQ, kDeqThreads);
          if (!ms.deq_ok) return;
        }
        uint16_t* dq = reinterpret_cast<uint16_t*>(smem + kOffDeq + (pass ? ds2 : ds) * kSlotBytes);
        for (int e = t * 16; e < kTileM * kKs; e += kDeqThreads * 16) {
          // e walks [k8][m8][8 rows][8 k]; 16 values are two rows of one core matrix
          const uint4 raw = *reinterpret_cast<const uint4*>(qv + e);
          const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
          uint32_t o8[8];
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int ee = e + h2 * 8;
            const int k8 = ee >> 10, m = ((ee >> 6) & 15) * 8 + ((ee >> 3) & 7);
            const __half2 d2 = __half2half2(sc[(k8 >> 2) * kTileM + m]);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              uint2 h, l;
              q8x4_to_f16x4_hilo(w4[h2 * 2 + i], d2, h, l);
              const uint2 v = pass ? l : h;
              o8[h2 * 4 + i * 2] = v.x; o8[h2 * 4 + i * 2 + 1] = v.y;
            }
          }
          *reinterpret_cast<uint4*>(dq + e) = make_uint4(o8[0], o8[1], o8[2], o8[3]);
          *reinterpret_cast<uint4*>(dq + e + 8) = make_uint4(o8[4], o8[5], o8[6], o8[7]);
        }
        fence_proxy_async_shared();
        named_bar(BAR_DEQ, kDeqThreads);
        if (t == 0) {
          if (pass == 1) mbar_arrive(&ms.wempty[rs]);
          mbar_arrive(&ms.dfull[pass ? ds2 : ds]);
        }
      }
    }
  }
}

// --------------------------------------------------------------- MMA warp
// Two-stage software pipeline over the CTA's slices: the operand copy of
// slice s+1 is issued (after its readiness counter is satisfied) before the
// MMAs of slice s, so operand latency overlaps tensor-core work.
__device__ void mma_role(const PParams& p, Misc& ms, uint8_t* smem) {
  uint32_t wit = 0, a_issue = 0, a_comp = 0, seg = 0;
  unsigned evi = 0;
  bool ok = true;
  for (int gi = 0; gi < p.NGEMM && ok; ++gi) {
    const GI G = gemm_inst(p, gi);
    const Ck c = chunking(G.R);
    int beg, end;
    my_run(c.n * G.n_mt, G.n_ks, gi, beg, end, p.det);
    const uint32_t idesc = idesc_f16(kTileM, c.Nc);
    const uint32_t abytes = uint32_t(kKs) * c.Nc * 2;
    const bool q8g = slice_is_q8(p, G);
    // Readiness of the run's operand slices: one batch of relaxed loads and a
    // single acquire fence up front, instead of an acquire round trip per slice.
    const int ch_lo = beg < end ? beg / G.n_ks / G.n_mt : 0;
    uint64_t seen = 0;
    if (beg < end) {
      const int ch_hi = (end - 1) / G.n_ks / G.n_mt;
      for (int ch = ch_lo; ch <= ch_hi; ++ch)
        for (int ks = 0; ks < G.n_ks; ++ks) {
          const int bit = (ch - ch_lo) * G.n_ks + ks;
          if (bit < 64 && ld_relaxed_u32(ready_cnt(p, gi, ch, ks)) >= unsigned(rows_in(G.R, c, ch)))
            seen |= 1ull << bit;
        }
      fence_acq_rel_gpu();
    }
    auto issue = [&](int s) -> bool {
      const int ks = s % G.n_ks, ch = s / G.n_ks / G.n_mt, bit = (ch - ch_lo) * G.n_ks + ks;
      if (!(bit < 64 && ((seen >> bit) & 1ull))) {
        if (!poll_geq(p, ready_cnt(p, gi, ch, ks), unsigned(rows_in(G.R, c, ch)))) return false;
        if (bit < 64) seen |= 1ull << bit;
      }
      ev_mma(p, evi, EV_READY, gi);
      const uint32_t a = a_issue % kNAct, au = a_issue / kNAct;
      if (au > 0 && !mwait(p, &ms.aempty[a], (au - 1) & 1)) return false;
      fence_proxy_async_global();
      mbar_expect_tx(&ms.afull[a], abytes);
      bulk_g2s(smem + kOffAct + a * kActBytes, G.act + size_t(ch) * G.Kdim * c.Nc + size_t(ks) * kKs * c.Nc, abytes,
               &ms.afull[a]);
      ++a_issue;
      return true;
    };
    if (beg < end && !issue(beg)) { ok = false; break; }
    for (int s = beg; s < end; ++s) {
      if (s + 1 < end && !issue(s + 1)) { ok = false; break; }
      const int ks = s % G.n_ks;
      const bool first = s == beg || ks == 0;
      const bool last = s == end - 1 || ks == G.n_ks - 1;
      const uint32_t a = a_comp % kNAct, au = a_comp / kNAct;
      // the weight images of the slice: one f16 image, or (Q8_0) the pair
      // hi, lo in two consecutive dequantised places, both multiplied into
      // the same accumulator
      const uint8_t* A[2];
      uint64_t* wfree[2];
      int nA = 1;
      if (tq8(p)) {
        // the first image now; a Q8_0 slice's lo image is waited for after
        // the hi image's MMAs are issued
        nA = q8g ? 2 : 1;
        for (int i = 0; i < nA; ++i) {
          const uint32_t ds = (wit + i) % kNDeq;
          A[i] = smem + kOffDeq + ds * kSlotBytes;
          wfree[i] = &ms.dempty[ds];
        }
        if (!mwait(p, &ms.dfull[wit % kNDeq], (wit / kNDeq) & 1)) { ok = false; break; }
      } else {
        const uint32_t ws = wit % kNSlotF16;
        if (!mwait(p, &ms.wfull[ws], (wit / kNSlotF16) & 1)) { ok = false; break; }
        A[0] = smem + kOffRing + ws * kSlotBytes;
        wfree[0] = &ms.wempty[ws];
      }
      ev_mma(p, evi, EV_WEIGHTS, gi);
      const uint32_t tb = seg & 1;
      if (first && seg >= 2 && !mwait(p, &ms.accempty[tb], ((seg >> 1) - 1) & 1)) { ok = false; break; }
      if (!mwait(p, &ms.afull[a], au & 1)) { ok = false; break; }
      ev_mma(p, evi, EV_LANDED, gi);
      tc_fence_after();
      const uint32_t b0 = smem_u32(smem + kOffAct + a * kActBytes), d = ms.tmem_base + tb * 128;
      for (int i = 0; i < nA; ++i) {
        if (i > 0) {
          if (!mwait(p, &ms.dfull[(wit + i) % kNDeq], ((wit + i) / kNDeq) & 1)) { ok = false; break; }
          tc_fence_after();
        }
        const uint32_t a0 = smem_u32(A[i]);
#pragma unroll
        for (int j = 0; j < kKs / 16; ++j) {
          const uint64_t ad = smem_desc(a0 + j * 2 * (kTileM / 8) * 128, (kTileM / 8) * 128, 128);
          const uint64_t bd = smem_desc(b0 + j * 2 * (c.Nc / 8) * 128, (c.Nc / 8) * 128, 128);
          mma_f16(d, ad, bd, idesc, (first && i == 0 && j == 0) ? 0u : 1u);
        }
        mma_commit(wfree[i]);   // the image's place is free once these MMAs complete
      }
      if (!ok) break;
      mma_commit(&ms.aempty[a]);
      if (last) {
        mma_commit(&ms.accfull[tb]);
        // second arrival, by this thread: releases (CTA scope) what its
        // acquires of the operand counters saw to the consumers' epilogue
        mbar_arrive(&ms.accfull[tb]);
        ev_mma(p, evi, EV_COMMIT, gi);
        ++seg;
      }
      wit += nA;
      ++a_comp;
    }
  }
  // every MMA retires, and every operand copy lands, before TMEM and shared
  // memory are released
  mma_commit(&ms.mmadone);
  mbar_wait(&ms.mmadone, 0);
  for (uint32_t k = a_comp; k < a_issue; ++k) mbar_wait(&ms.afull[k % kNAct], (k / kNAct) & 1);
}

// ------------------------------------------------------ consumer helpers
// Step-1 inputs, one warp per row r < 2B: operand rows 2b = f16(H_b),
// 2b+1 = f16(E0[q0_b]); residual rows start at the projection bias.
__device__ bool prep1_items(const PParams& p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, G = gridDim.x;
  const int R = 2 * p.B;
  const Ck c = chunking(R);
  for (int r = blockIdx.x + warp * G; r < R; r += kConsumerWarps * G) {
    const int b = r >> 1, ch = r / c.Nc;
    constexpr int kG = 8;   // loads in flight per lane before the stores
    if ((r & 1) == 0) {
      // the row's range exponent from its mean square; the projection's
      // output (and so layer 0's QKV operand of this row) takes the same
      const float* hr = p.H + size_t(b) * p.th;
      float ss = 0.f;
      for (int k0 = lane * 4; k0 < p.th; k0 += 128 * kG) {
        float4 hv[kG];
#pragma unroll
        for (int i = 0; i < kG; ++i)
          hv[i] = k0 + i * 128 < p.th ? __ldg(reinterpret_cast<const float4*>(hr + k0 + i * 128))
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < kG; ++i) ss += hv[i].x * hv[i].x + hv[i].y * hv[i].y + hv[i].z * hv[i].z + hv[i].w * hv[i].w;
      }
      const int e = range_exp(warp_sum(ss) / float(p.th));
      const float sc = exp2i(-e);
      if (lane == 0) {
        *rexp_at(p, 0, r) = e;
        *rexp_at(p, gi_of(p, 1, 0, 0), r) = e;
      }
      for (int k0 = lane * 4; k0 < p.th; k0 += 128 * kG) {
        float4 hv[kG];
#pragma unroll
        for (int i = 0; i < kG; ++i)
          hv[i] = k0 + i * 128 < p.th ? __ldg(reinterpret_cast<const float4*>(hr + k0 + i * 128))
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < kG; ++i) {
          if (k0 + i * 128 >= p.th) break;
          *reinterpret_cast<uint2*>(p.a1[0] + act_off(r, k0 + i * 128, p.th, c)) =
              pack4_f16(hv[i].x * sc, hv[i].y * sc, hv[i].z * sc, hv[i].w * sc);
        }
      }
    } else {
      int q = p.q0[b];
      if (q < 0 || q >= p.q0_vocab) {
        if (lane == 0) set_status(p.status, QP_ERR_BAD_TOKEN);
        q = q < 0 ? 0 : p.q0_vocab - 1;
      }
      for (int k0 = lane * 4; k0 < p.th; k0 += 128 * kG) {
        uint2 ev[kG];
#pragma unroll
        for (int i = 0; i < kG; ++i)
          ev[i] = k0 + i * 128 < p.th ? __ldg(reinterpret_cast<const uint2*>(p.e0 + size_t(q) * p.th + k0 + i * 128))
                                      : make_uint2(0, 0);
#pragma unroll
        for (int i = 0; i < kG; ++i) {
          if (k0 + i * 128 >= p.th) break;
          *reinterpret_cast<uint2*>(p.a1[0] + act_off(r, k0 + i * 128, p.th, c)) =
              pack4_f16(e16_to_f32(ev[i].x, p.embed_f16), e16_to_f32(ev[i].x >> 16, p.embed_f16),
                        e16_to_f32(ev[i].y, p.embed_f16), e16_to_f32(ev[i].y >> 16, p.embed_f16));
        }
      }
    }
    for (int kk = lane * 4; kk < p.d; kk += 128)
      *reinterpret_cast<float4*>(p.x1 + size_t(r) * p.d + kk) = *reinterpret_cast<const float4*>(p.b_proj + kk);
    __syncwarp();
    if (lane == 0) {
      fence_acq_rel_gpu();   // one fence releases the row for every slice count below
      for (int ks = 0; ks < p.th / kKs; ++ks) red_relaxed_add(ready_cnt(p, 0, ch, ks), 1);
    }
  }
  return true;
}

// The code of step `step` for frame b (lane 0 only): waits for the argmax or
// the sampled decision.  Returns -1 if the grid aborted.
__device__ int wait_code(const PParams& p, int step, int b) {
  const Ck c = chunking(p.B);
  if (p.temperature > 0.f) {
    unsigned* dp = p.decided + size_t(step - 1) * p.B + b;
    if (!poll_geq(p, dp, 1u)) return -1;
    return int(ld_acquire_u32(dp)) - 1;
  }
  if (!poll_geq(p, head_done(p, step, b / c.Nc), unsigned(p.V / kTileM))) return -1;
  return unpack_argmax_index(ld_acquire_u64(p.codepk + size_t(step - 1) * p.B + b));
}

// Step k >= 2 inputs, one warp per frame: report the previous step's code,
// embed the next input (teacher-forced if asked) as residual row b and as
// the layer-0 QKV operand f16(E * w_attn_norm); its squared norm comes from
// the table precomputed at load.
__device__ bool prepk_items(const PParams& p, int k) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, G = gridDim.x;
  const Ck c = chunking(p.B);
  const int gi = gi_of(p, k, 0, 0);
  const float* wn = p.layer[0].attn_norm;
  for (int b = (blockIdx.x + k * 11) % G + warp * G; b < p.B; b += kConsumerWarps * G) {
    int nc = 0;
    if (lane == 0) {
      const int code = wait_code(p, k - 1, b);
      if (code >= 0) {
        p.out_codes[size_t(b) * p.n_steps + (k - 2)] = code;
        nc = p.forced ? p.forced[size_t(b) * p.n_steps + (k - 2)] : code;
        if (nc < 0 || nc >= p.V) {
          set_status(p.status, QP_ERR_BAD_TOKEN);
          nc = nc < 0 ? 0 : p.V - 1;
        }
      } else {
        nc = -1;
      }
    }
    nc = __shfl_sync(0xffffffffu, nc, 0);
    if (nc < 0) return false;
    __syncwarp();   // the writes below follow lane 0's acquire
    if (p.proj_in) {
      // Talker-wide table: row b of the step's projection operand is
      // f16(E[k-2][nc]); the residual row starts at the projection's bias
      const int gp = gi_proj(p, k);
      const uint16_t* e = p.embed[k - 2] + size_t(nc) * p.th;
      constexpr int kG = 8;   // loads in flight per lane before the stores
      for (int k0 = lane * 4; k0 < p.th; k0 += 128 * kG) {
        uint2 ev[kG];
#pragma unroll
        for (int i = 0; i < kG; ++i)
          ev[i] = k0 + i * 128 < p.th ? __ldg(reinterpret_cast<const uint2*>(e + k0 + i * 128)) : make_uint2(0, 0);
#pragma unroll
        for (int i = 0; i < kG; ++i) {
          if (k0 + i * 128 >= p.th) break;
          *reinterpret_cast<uint2*>(p.a1[0] + act_off(b, k0 + i * 128, p.th, c)) =
              pack4_f16(e16_to_f32(ev[i].x, p.embed_f16), e16_to_f32(ev[i].x >> 16, p.embed_f16),
                        e16_to_f32(ev[i].y, p.embed_f16), e16_to_f32(ev[i].y >> 16, p.embed_f16));
        }
      }
      for (int kk = lane * 4; kk < p.d; kk += 128)
        *reinterpret_cast<float4*>(p.xk + size_t(b) * p.d + kk) = *reinterpret_cast<const float4*>(p.b_proj + kk);
      __syncwarp();
      if (lane == 0) {
        const int ch = b / c.Nc;
        fence_acq_rel_gpu();   // one fence releases the row for every slice count below
        for (int ks = 0; ks < p.th / kKs; ++ks) red_relaxed_add(ready_cnt(p, gp, ch, ks), 1);
      }
      continue;
    }
    const uint16_t* e = p.embed[k - 2] + size_t(nc) * p.d;
    // the row's loads all in flight before its stores (a store could alias a
    // later load, so the compiler keeps a fused loop's loads in order)
    constexpr int kG = 8;   // 1024 columns per pass
    for (int k0 = lane * 4; k0 < p.d; k0 += 128 * kG) {
      uint2 ev[kG];
      float4 wv[kG];
#pragma unroll
      for (int i = 0; i < kG; ++i) {
        const int kk = k0 + i * 128;
        ev[i] = kk < p.d ? __ldg(reinterpret_cast<const uint2*>(e + kk)) : make_uint2(0, 0);
        wv[i] = kk < p.d ? __ldg(reinterpret_cast<const float4*>(wn + kk)) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int i = 0; i < kG; ++i) {
        const int kk = k0 + i * 128;
        if (kk >= p.d) break;
        const float v0 = e16_to_f32(ev[i].x, p.embed_f16), v1 = e16_to_f32(ev[i].x >> 16, p.embed_f16);
        const float v2 = e16_to_f32(ev[i].y, p.embed_f16), v3 = e16_to_f32(ev[i].y >> 16, p.embed_f16);
        *reinterpret_cast<float4*>(p.xk + size_t(b) * p.d + kk) = make_float4(v0, v1, v2, v3);
        const float4 w = wv[i];
        *reinterpret_cast<uint2*>(p.ak[0] + act_off(b, kk, p.d, c)) =
            pack4_f16(v0 * w.x, v1 * w.y, v2 * w.z, v3 * w.w);
      }
    }
    if (lane == 0) {
      if (!p.det) {
        *ss_at(p, gi, b) = p.embed_ss[k - 2][nc];
      } else {
        for (int mt = 0; mt < p.d / kTileM; ++mt) *ss_part_at(p, gi, mt, b) = mt == 0 ? p.embed_ss[k - 2][nc] : 0.f;
      }
    }
    __syncwarp();
    if (lane == 0) {
      const int ch = b / c.Nc;
      fence_acq_rel_gpu();   // one fence releases the row for every count below
      for (int ks = 0; ks < p.d / kKs; ++ks) red_relaxed_add(ready_cnt(p, gi, ch, ks), 1);
      red_relaxed_add(ss_cnt(p, gi, ch), unsigned(p.d / kTileM));
    }
  }
  return true;
}

__device__ bool final_items(const PParams& p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, G = gridDim.x;
  for (int b = (blockIdx.x + 5) % G + warp * G; b < p.B; b += kConsumerWarps * G) {
    int code = 0;
    if (lane == 0) {
      code = wait_code(p, p.n_steps, b);
      if (code >= 0) p.out_codes[size_t(b) * p.n_steps + (p.n_steps - 1)] = code;
    }
    code = __shfl_sync(0xffffffffu, code, 0);
    if (code < 0) return false;
  }
  return true;
}

// Attention of one (frame, kv head) per warp at layer l of step k: per-head
// norms and RoPE of the new position(s), KV append, causal softmax over
// positions 0..pos for the group's q heads; output into the O operand.
// Lane l holds dims 4l..4l+3 of every 128-vector.  Scores of two q heads x
// 16 positions are 32 partial dot products per lane, summed across the warp
// by one reduce-scatter that leaves score (head l/16, position l%16) in lane l.
__device__ bool attn_items(const PParams& p, Misc& ms, int k, int l) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, G = gridDim.x;
  const int P = k == 1 ? 2 : 1, pos0 = k == 1 ? 0 : k, R = p.B * P;
  const Ck c = chunking(R);
  const int gi_q = gi_of(p, k, l, 0), gi_o = gi_q + 1;
  const int qkvw = p.qw + 2 * p.kvw, grp = p.n_q / p.n_kv, ctx = p.n_steps + 1;
  float* acc = k == 1 ? p.acc1_qkv : p.acck_qkv;
  uint16_t* act_o = k == 1 ? p.a1[2] : p.ak[1];
  const PLayer& L = p.layer[l];
  const int n_items = p.B * p.n_kv, nks = p.d / kKs;
  const float scale = rsqrtf(128.f);
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  uint16_t* kvl = p.kv + size_t(l) * p.Bmax * ctx * 2 * p.kvw;
  // Each warp takes a contiguous range of items in (kv head, frame) order, so
  // that consecutive items of one kv head and one 128-row chunk form a group:
  // one readiness poll before the group, one release of its rows after it.
  const int gw = warp * G + (blockIdx.x + gi_q * 13) % G, W = kConsumerWarps * G;
  const int i_beg = int((long long)n_items * gw / W), i_end = int((long long)n_items * (gw + 1) / W);
  int g_j = -1, g_ch = -1, g_rows = 0;   // the open group
  auto close_group = [&]() {
    __syncwarp();   // every lane's writes precede lane 0's release
    if (lane == 0 && g_rows > 0)
      for (int g2 = 0; g2 < grp; ++g2) red_release_add(ready_cnt(p, gi_o, g_ch, g_j * grp + g2), unsigned(g_rows));
    g_rows = 0;
  };
  for (int i = i_beg; i < i_end; ++i) {
    const int j = i / p.B, b = i % p.B, r0 = b * P, ch = r0 / c.Nc;
    if (j != g_j || ch != g_ch) {
      close_group();
      g_j = j;
      g_ch = ch;
      // the group's q tiles, its k tile and its v tile: one lane polls each
      int okl = 1;
      if (lane < grp + 2) {
        const int tile = lane < grp ? j * grp + lane
                                    : (lane == grp ? p.qw / kTileM + j : (p.qw + p.kvw) / kTileM + j);
        okl = poll_geq(p, tile_cnt(p, gi_q, ch, tile), unsigned(nks));
      }
      if (!__all_sync(0xffffffffu, okl)) return false;
      __syncwarp();   // order every lane's reads after the acquires
    }
    if (lane == 0) ev_cons(p, &ms.evc, EV_ATT_READY, gi_q);
    uint16_t* kvb = kvl + size_t(b) * ctx * 2 * p.kvw + j * 128 + lane * 4;   // + (pos*2 + {0,1}) * kvw
    for (int pp = 0; pp < P; ++pp) {
      const int r = r0 + pp, pos = pos0 + pp;
      float* row = acc + size_t(r) * qkvw;
      float* kr = row + p.qw + j * 128 + lane * 4;
      float* vr = row + p.qw + p.kvw + j * 128 + lane * 4;
      // every load of the item that does not depend on another is issued first:
      // the new k, v and the first two q heads, then the cached keys and values
      const float4 kraw = __ldcg(reinterpret_cast<const float4*>(kr));
      const float4 vnew = __ldcg(reinterpret_cast<const float4*>(vr));
      float4 qraw[2];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
        qraw[hh] = hh < grp ? __ldcg(reinterpret_cast<const float4*>(row + (j * grp + hh) * 128 + lane * 4)) : z4;
      uint2 kh[kMaxCtx], vh[kMaxCtx];
#pragma unroll
      for (int t = 0; t < kMaxCtx; ++t) {
        kh[t] = t < pos ? __ldcg(reinterpret_cast<const uint2*>(kvb + (size_t(t) * 2 + 0) * p.kvw)) : make_uint2(0, 0);
        vh[t] = t < pos ? __ldcg(reinterpret_cast<const uint2*>(kvb + (size_t(t) * 2 + 1) * p.kvw)) : make_uint2(0, 0);
      }
      const float4 knew = norm_rope(kraw, L.k_norm, p.eps, p.rope_cs + pos * 64, lane);
      *reinterpret_cast<uint2*>(kvb + (size_t(pos) * 2 + 0) * p.kvw) = pack4_f16(knew.x, knew.y, knew.z, knew.w);
      *reinterpret_cast<uint2*>(kvb + (size_t(pos) * 2 + 1) * p.kvw) = pack4_f16(vnew.x, vnew.y, vnew.z, vnew.w);
      *reinterpret_cast<float4*>(kr) = z4;
      *reinterpret_cast<float4*>(vr) = z4;
      for (int g0 = 0; g0 < grp; g0 += 2) {
        const int nh = min(2, grp - g0);
        float4 qn[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          qn[hh] = z4;
          if (hh < nh) {
            float* qr = row + (j * grp + g0 + hh) * 128 + lane * 4;
            const float4 q = g0 == 0 ? qraw[hh] : __ldcg(reinterpret_cast<const float4*>(qr));
            qn[hh] = norm_rope(q, L.q_norm, p.eps, p.rope_cs + pos * 64, lane);
            *reinterpret_cast<float4*>(qr) = z4;
          }
        }
        float part[32];
#pragma unroll
        for (int t = 0; t < kMaxCtx; ++t) {
          const float4 kk = t < pos ? unpack4_f16(kh[t]) : (t == pos ? knew : z4);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
            part[hh * 16 + t] = qn[hh].x * kk.x + qn[hh].y * kk.y + qn[hh].z * kk.z + qn[hh].w * kk.w;
        }
        // lane l: score of head (l >> 4), position (l & 15)
        const bool valid = (lane >> 4) < nh && (lane & 15) <= pos;
        const float rsum = reduce_scatter32(part, lane);   // all 32 lanes take part
        const float sc = valid ? rsum * scale : -INFINITY;
        float mx = sc;
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float e = valid ? expf(sc - mx) : 0.f;
        float den = e;
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
        const float pr = den > 0.f ? e / den : 0.f;
        float4 o2[2] = {z4, z4};
#pragma unroll
        for (int t = 0; t < kMaxCtx; ++t) {
          const float4 vv = t < pos ? unpack4_f16(vh[t]) : (t == pos ? vnew : z4);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const float w = __shfl_sync(0xffffffffu, pr, hh * 16 + t);
            o2[hh].x += w * vv.x; o2[hh].y += w * vv.y; o2[hh].z += w * vv.z; o2[hh].w += w * vv.w;
          }
        }
        for (int hh = 0; hh < nh; ++hh)
          *reinterpret_cast<uint2*>(act_o + act_off(r, (j * grp + g0 + hh) * 128 + lane * 4, p.qw, c)) =
              pack4_f16(o2[hh].x, o2[hh].y, o2[hh].z, o2[hh].w);
      }
      __syncwarp();   // the next position of this frame reads what was stored here
    }
    g_rows += P;
    if (lane == 0) ev_cons(p, &ms.evc, EV_ATT_DONE, gi_q);
  }
  close_group();
  return true;
}

// Finishing work of rows [lo, hi) of a completed tile (all consumer threads
// of one of the tile's contributing CTAs; the contributors split the rows).
// Each warp takes rows lo + warp, lo + warp + 8, ...; the loads of several
// of its rows are issued together.
template <int KIND>
__device__ bool finish_rows(const PParams& p, Misc& ms, const GI& G, int gi, int ch, int mt, Ck c, int lo, int hi) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  if (KIND == G_QKV) return true;
  if (KIND == G_PROJ || KIND == G_O || KIND == G_DOWN) {
    const float* X = G.acc;
    const int feat = mt * kTileM + lane * 4;
    bool to_head = false;
    int gi_n;
    const float* w;
    uint16_t* act_n;
    if (KIND == G_PROJ) {
      gi_n = gi_of(p, G.k, 0, 0); w = p.layer[0].attn_norm; act_n = G.k == 1 ? p.a1[1] : p.ak[0];
    } else if (KIND == G_O) {
      gi_n = gi + 1; w = p.layer[G.l].ffn_norm; act_n = G.k == 1 ? p.a1[3] : p.ak[2];
    } else if (G.l + 1 < p.L) {
      gi_n = gi + 1; w = p.layer[G.l + 1].attn_norm; act_n = G.k == 1 ? p.a1[1] : p.ak[0];
    } else {
      to_head = true; gi_n = gi_head(p, G.k); w = p.out_norm; act_n = p.ahead;
    }
    const float4 wv = *reinterpret_cast<const float4*>(w + feat);
    const int P = G.k == 1 ? 2 : 1;
    const Ck ch_h = chunking(p.B);
    // The range exponent of each row of the next operand: from the mean
    // square of the row as it entered this GEMM's sublayer (the QKV input
    // for O, the gate/up input for down), which is complete; for the
    // projection, the one the step-1 input pass chose from H (0 for table
    // rows).  Every tile of a row computes the same exponent; tile 0 records it.
    auto row_exp = [&](int n) -> int {
      if (KIND == G_PROJ) return G.k == 1 ? __ldcg(rexp_at(p, gi_n, n)) : 0;
      return range_exp(ss_total(p, gi - 1, n) / float(p.d));
    };
    for (int r0 = lo + warp; r0 < hi; r0 += 8 * kConsumerWarps) {
      float4 xv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int row = r0 + u * kConsumerWarps, n = ch * c.Nc + row;
        const bool use = row < hi && (!to_head || (n % P) == P - 1);
        xv[u] = use ? __ldcg(reinterpret_cast<const float4*>(X + size_t(n) * p.d + feat)) : z4;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int row = r0 + u * kConsumerWarps, n = ch * c.Nc + row;
        if (row >= hi || (to_head && (n % P) != P - 1)) continue;
        const float4 x = xv[u];
        const float sq = warp_sum(x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w);
        const int nr = to_head ? n / P : n;
        const int e = row_exp(n);
        const float sc = exp2i(-e);
        if (lane == 0) {
          if (p.det) *ss_part_at(p, gi_n, mt, nr) = sq;
          else red_add_f32(ss_at(p, gi_n, nr), sq);
          if (mt == 0 && KIND != G_PROJ) *rexp_at(p, gi_n, nr) = e;
        }
        *reinterpret_cast<uint2*>(act_n + act_off(nr, feat, p.d, to_head ? ch_h : c)) =
            pack4_f16(x.x * wv.x * sc, x.y * wv.y * sc, x.z * wv.z * sc, x.w * wv.w * sc);
      }
    }
    named_bar(BAR_CONS, kConsumers);
    if (t == 0 && hi > lo) {
      // release: the bar.sync above orders every consumer thread's writes first
      fence_acq_rel_gpu();   // one fence releases the rows for every count below
      if (!to_head) {
        red_relaxed_add(ready_cnt(p, gi_n, ch, mt), unsigned(hi - lo));
        red_relaxed_add(ss_cnt(p, gi_n, ch), unsigned(hi - lo));
      } else {
        // frames whose last position lies in these rows: [nlo/P, nhi/P)
        const int f0 = (ch * c.Nc + lo) / P, f1 = (ch * c.Nc + hi) / P;
        for (int hc = f0 / ch_h.Nc; f1 > f0 && hc <= (f1 - 1) / ch_h.Nc; ++hc) {
          const int lo = max(f0, hc * ch_h.Nc), hi = min(f1, (hc + 1) * ch_h.Nc);
          red_relaxed_add(ready_cnt(p, gi_n, hc, mt), unsigned(hi - lo));
          red_relaxed_add(ss_cnt(p, gi_n, hc), unsigned(hi - lo));
        }
      }
    }
    return true;
  }
  if (KIND == G_GU) {
    // mt is the pair's gate tile: gate|up tiles mt and F/128 + mt hold
    // columns 128 mt .. +127 of gate and of up
    const int kd = mt;
    uint16_t* act_d = G.k == 1 ? p.a1[4] : p.ak[3];
    const int feat = kd * kTileM + lane * 4;
    for (int r0 = lo + warp; r0 < hi; r0 += 4 * kConsumerWarps) {
      float4 gv[4], uv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int row = r0 + u * kConsumerWarps;
        const float* gp = G.acc + size_t(ch * c.Nc + row) * 2 * p.F + feat;
        gv[u] = row < hi ? __ldcg(reinterpret_cast<const float4*>(gp)) : z4;
        uv[u] = row < hi ? __ldcg(reinterpret_cast<const float4*>(gp + p.F)) : z4;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int row = r0 + u * kConsumerWarps, n = ch * c.Nc + row;
        if (row >= hi) continue;
        float* gp = G.acc + size_t(n) * 2 * p.F + feat;
        const float4 g = gv[u], uu = uv[u];
        *reinterpret_cast<uint2*>(act_d + act_off(n, feat, p.F, c)) =
            pack4_f16(silu_f(g.x) * uu.x, silu_f(g.y) * uu.y, silu_f(g.z) * uu.z, silu_f(g.w) * uu.w);
        *reinterpret_cast<float4*>(gp) = z4;
        *reinterpret_cast<float4*>(gp + p.F) = z4;
      }
    }
    named_bar(BAR_CONS, kConsumers);
    if (t == 0 && hi > lo) red_release_add(ready_cnt(p, gi + 1, ch, kd), unsigned(hi - lo));
    return true;
  }
  // G_HEAD: final logits of 128 codebook entries for the chunk's frames
  {
    const int col = mt * kTileM + lane * 4;
    const bool greedy = p.temperature <= 0.f;
    for (int r0 = lo + warp; r0 < hi; r0 += 4 * kConsumerWarps) {
      float4 lv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int row = r0 + u * kConsumerWarps;
        lv[u] = row < hi ? __ldcg(reinterpret_cast<const float4*>(p.logits + size_t(ch * c.Nc + row) * p.V + col)) : z4;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int row = r0 + u * kConsumerWarps, b = ch * c.Nc + row;
        if (row >= hi) continue;
        const float4 lg = lv[u];
        if (p.out_logits)
          *reinterpret_cast<float4*>(p.out_logits + (size_t(b) * p.n_steps + (G.k - 1)) * p.V + col) = lg;
        if (greedy) {
          unsigned long long best = pack_argmax(lg.x, col);
          const unsigned long long c1 = pack_argmax(lg.y, col + 1), c2 = pack_argmax(lg.z, col + 2),
                                   c3 = pack_argmax(lg.w, col + 3);
          best = c1 > best ? c1 : best;
          best = c2 > best ? c2 : best;
          best = c3 > best ? c3 : best;
          best = warp_max_u64(best);
          if (lane == 0) atomicMax(p.codepk + size_t(G.k - 1) * p.B + b, best);
          *reinterpret_cast<float4*>(p.logits + size_t(b) * p.V + col) = z4;
        }
      }
    }
    named_bar(BAR_CONS, kConsumers);
    if (t == 0 && hi > lo) {
      // the tile counter counts the finished rows past its K slices: the
      // share that completes the tile's rows counts the tile done
      const unsigned add = unsigned(hi - lo), full = unsigned(G.n_ks) + unsigned(rows_in(G.R, c, ch));
      if (atom_add_acq_rel(tile_cnt(p, gi, ch, mt), add) + add == full) red_release_add(head_done(p, G.k, ch), 1u);
    }
    return true;
  }
}

// Drain this CTA's accumulator segments of GEMM gi.
template <int KIND>
__device__ bool epilogues(const PParams& p, Misc& ms, uint32_t* keys, int gi, uint32_t& seg) {
  const GI G = gemm_inst(p, gi);
  const Ck c = chunking(G.R);
  int beg, end;
  my_run(c.n * G.n_mt, G.n_ks, gi, beg, end, p.det);
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const bool scaled = KIND == G_QKV || KIND == G_GU || KIND == G_HEAD;
  int s = beg;
  while (s < end) {
    const int ks = s % G.n_ks, tt = s / G.n_ks, mt = tt % G.n_mt, ch = tt / G.n_mt;
    const int seg_end = min(end, s + (G.n_ks - ks)), nsl = seg_end - s;
    const uint32_t tb = seg & 1;
    const int rows = rows_in(G.R, c, ch);
    // consumer-wide waits are taken by thread 0 and broadcast, so that every
    // consumer thread leaves (or stays) together.  The norm statistics of a
    // scaled GEMM are gathered first, while the MMAs may still run.
    // Each row's factor: 1/RMS of the normalised input times 2^e, which
    // undoes the operand's range scaling 2^-e.
    if (scaled) {
      if (t == 0) ms.flag[1] = poll_geq(p, ss_cnt(p, gi, ch), unsigned(rows * (p.d / kTileM)));
      named_bar(BAR_CONS, kConsumers);
      if (!ms.flag[1]) return false;
      for (int col = t; col < c.Nc; col += kConsumers) {
        const int n = ch * c.Nc + col;
        ms.inv[col] = n < G.R ? rsqrtf(ss_total(p, gi, n) / float(p.d) + p.eps) * exp2i(__ldcg(rexp_at(p, gi, n)))
                              : 0.f;
      }
    }
    if (t == 0) ms.flag[1] = mwait(p, &ms.accfull[tb], (seg >> 1) & 1);
    named_bar(BAR_CONS, kConsumers);
    if (!ms.flag[1]) return false;
    if (t == 0) ev_cons(p, &ms.evc, EV_ACC, gi);
    tc_fence_after();
    // Each warp drains 32 accumulator rows (features) x 8 columns (frames) at
    // a time, transposes them through its 1 KB of shared memory, and adds 4
    // consecutive features per thread with one vector reduction.
    const int quarter = warp & 3, half = warp >> 2, cols = c.Nc / 2;
    const int m0 = mt * kTileM + quarter * 32;
    float* tp = reinterpret_cast<float*>(keys) + warp * 256;   // [8 frames][32 features]
    for (int col = half * cols; col < (half + 1) * cols; col += 8) {
      float v[8];
      tmem_ld8(ms.tmem_base + tb * 128 + (uint32_t(quarter * 32) << 16) + uint32_t(col), v);
#pragma unroll
      for (int i = 0; i < 8; ++i) tp[i * 32 + lane] = v[i];
      __syncwarp();
#pragma unroll
      for (int pass = 0; pass < 2; ++pass) {
        const int f = pass * 4 + (lane >> 3), k4 = (lane & 7) * 4, n = ch * c.Nc + col + f;
        if (n < G.R) {
          float4 x = *reinterpret_cast<const float4*>(tp + f * 32 + k4);
          if (scaled || KIND == G_PROJ) {
            // the projection's factor is read here, after the accumulator
            // wait, which orders it after the step-1 input passes of every
            // row of the chunk (they publish the rows' exponents)
            const float s = scaled ? ms.inv[col + f] : (G.k == 1 ? exp2i(__ldcg(rexp_at(p, gi, n))) : 1.f);
            x.x *= s; x.y *= s; x.z *= s; x.w *= s;
          }
          red_add_v4_f32(G.acc + size_t(n) * G.ld + m0 + k4, x);
        }
      }
      __syncwarp();
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&ms.accempty[tb]);
    named_bar(BAR_CONS, kConsumers);
    if (t == 0) {
      ev_cons(p, &ms.evc, EV_REDS, gi);
      // release: the bar.sync above orders every consumer thread's reductions first
      // (a test of the failure path makes one count go missing)
      if (!(gi == p.withhold && beg == 0 && s == beg)) red_release_add(tile_cnt(p, gi, ch, mt), unsigned(nsl));
      ev_cons(p, &ms.evc, EV_COUNTED, gi);
    }
    ++seg;
    s = seg_end;
  }
  if (KIND == G_QKV || beg >= end) return true;   // attention items read the QKV tiles as they complete
  // The finishing passes of the tiles this CTA added into, once every
  // contribution is in: the tile's contributors split its rows, so a pass
  // takes a fraction of one CTA's time.  All of this CTA's drains precede
  // these waits, and every contributor drains before it waits, so each wait
  // ends.  A gate|up pair (gate tile kd, up tile F/128 + kd) is finished by
  // the contributors of both.
  const int tiles = c.n * G.n_mt;
  for (int tt = beg / G.n_ks; tt <= (end - 1) / G.n_ks; ++tt) {
    const int mt = tt % G.n_mt, ch = tt / G.n_mt, rows = rows_in(G.R, c, ch);
    int n = 0, rank = tile_share(tiles, G.n_ks, gi, tt, n, p.det), mt_f = mt;
    if (KIND == G_GU) {
      const int nkd = p.F / kTileM, kd = mt % nkd, tg = ch * G.n_mt + kd, tu = tg + nkd;
      int ng = 0, nu = 0;
      const int rg = tile_share(tiles, G.n_ks, gi, tg, ng, p.det), ru = tile_share(tiles, G.n_ks, gi, tu, nu, p.det);
      rank = mt < nkd ? rg : ng + ru;
      n = ng + nu;
      mt_f = kd;
      if (t == 0)
        ms.flag[1] = poll_geq(p, tile_cnt(p, gi, ch, kd), unsigned(G.n_ks)) &&
                     poll_geq(p, tile_cnt(p, gi, ch, kd + nkd), unsigned(G.n_ks));
    } else if (t == 0) {
      ms.flag[1] = poll_geq(p, tile_cnt(p, gi, ch, mt), unsigned(G.n_ks));
    }
    named_bar(BAR_CONS, kConsumers);
    if (!ms.flag[1]) return false;
    const int lo = int((long long)rows * rank / n), hi = int((long long)rows * (rank + 1) / n);
    if (!finish_rows<KIND>(p, ms, G, gi, ch, mt_f, c, lo, hi)) return false;
    if (t == 0) ev_cons(p, &ms.evc, EV_LASTDONE, gi);
  }
  return true;
}

// Gumbel top-k decisions of step k: each half of the consumer warps (4
// warps) decides one frame, so a CTA takes two frames at a time (one, by
// half 0, when the vocabulary is too large for two key arrays).
__device__ bool decide_items(const PParams& p, Misc& ms, uint32_t* keys, int k) {
  constexpr int NG = kConsumers / 2;
  const int V = p.V, t = threadIdx.x, G = gridDim.x, half = t / NG, tg = t - half * NG;
  const bool two = 2 * V <= kMaxVocab;
  const Ck c = chunking(p.B);
  const int bar = BAR_HALF0 + half;
  for (int b0 = (blockIdx.x + k * 7) % G; b0 < p.B; b0 += two ? 2 * G : G) {
    const int b = b0 + (two ? half * G : 0);
    if (b >= p.B || (!two && half == 1)) continue;   // warp-uniform: the half sits this frame out
    if (tg == 0) ms.hflag[half] = poll_geq(p, head_done(p, k, b / c.Nc), unsigned(V / kTileM));
    named_bar(bar, NG);
    if (!ms.hflag[half]) return false;
    if (tg == 0) ev_cons(p, &ms.evc, EV_DEC_READY, gi_head(p, k));
    float* l = p.logits + size_t(b) * V;
    const float* gb = p.gumbel + (size_t(b) * p.n_steps + (k - 1)) * V;
    const int code = gumbel_topk_group<NG>(l, 1.f, p.temperature, gb, V, p.top_k, keys + (two ? half * V : 0),
                                           ms.topk[half], bar, tg);
    for (int i = tg; i < V; i += NG) l[i] = 0.f;   // the buffer is reused next step
    named_bar(bar, NG);
    if (tg == 0) {
      __threadfence();
      atomicExch(p.decided + size_t(k - 1) * p.B + b, unsigned(code + 1));
      ev_cons(p, &ms.evc, EV_DEC_DONE, gi_head(p, k));
    }
  }
  return true;
}

#ifdef QP_TRACE
__device__ __forceinline__ void trace_mark(const PParams& p, int sec, int which) {
  if (p.trace && threadIdx.x == 0 && sec < p.trace_n)
    p.trace[(size_t(sec) * gridDim.x + blockIdx.x) * 2 + which] = globaltimer_ns();
}
#else
__device__ __forceinline__ void trace_mark(const PParams&, int, int) {}
#endif

__device__ void consumer_role(const PParams& p, Misc& ms, uint8_t* smem) {
  uint32_t seg = 0;
  int sec = 0;
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + kOffKeys);
  // A section ends with one consumer-wide barrier; a failed wait in any warp
  // makes every consumer warp leave there together.
#define QP_SECTION(expr)                      \
  {                                           \
    trace_mark(p, sec, 0);                    \
    const bool ok_ = (expr);                  \
    if (!ok_) ms.fail = 1;                    \
    named_bar(BAR_CONS, kConsumers);          \
    trace_mark(p, sec, 1);                    \
    ++sec;                                    \
    if (ms.fail) return;                      \
  }
  QP_SECTION(prep1_items(p));
  for (int k = 1; k <= p.n_steps; ++k) {
    if (k > 1) QP_SECTION(prepk_items(p, k));
    // one call site: a section inlined twice costs instruction fetch
    if (k == 1 || p.proj_in) QP_SECTION(epilogues<G_PROJ>(p, ms, keys, gi_proj(p, k), seg));
    for (int l = 0; l < p.L; ++l) {
      QP_SECTION(epilogues<G_QKV>(p, ms, keys, gi_of(p, k, l, 0), seg));
      QP_SECTION(attn_items(p, ms, k, l));
      QP_SECTION(epilogues<G_O>(p, ms, keys, gi_of(p, k, l, 1), seg));
      QP_SECTION(epilogues<G_GU>(p, ms, keys, gi_of(p, k, l, 2), seg));
      QP_SECTION(epilogues<G_DOWN>(p, ms, keys, gi_of(p, k, l, 3), seg));
    }
    QP_SECTION(epilogues<G_HEAD>(p, ms, keys, gi_head(p, k), seg));
    if (p.temperature > 0.f) QP_SECTION(decide_items(p, ms, keys, k));
  }
  QP_SECTION(final_items(p));
#undef QP_SECTION
}

#if QP_TILE_Q8
#define TILE_KERNEL k_frames_q8
#else
#define TILE_KERNEL k_frames
#endif
__global__ void __launch_bounds__(kThreads, 1) TILE_KERNEL(const PParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Misc& ms = *reinterpret_cast<Misc*>(smem + kOffMisc);
  const int t = threadIdx.x, warp = t >> 5;
  if (t == 0) {
    for (int i = 0; i < kNSlotF16; ++i) { mbar_init(&ms.wfull[i], 1); mbar_init(&ms.wempty[i], 1); }
    for (int i = 0; i < kNDeq; ++i) { mbar_init(&ms.dfull[i], 1); mbar_init(&ms.dempty[i], 1); }
    for (int i = 0; i < kNAct; ++i) { mbar_init(&ms.afull[i], 1); mbar_init(&ms.aempty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&ms.accfull[i], 2); mbar_init(&ms.accempty[i], kConsumerWarps); }
    mbar_init(&ms.mmadone, 1);
    ms.fail = 0;
    ms.deq_ok = 1;
    ms.evc = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(&ms.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp < kConsumerWarps) {
    consumer_role(p, ms, smem);
  } else if (warp == kProducerWarp) {
    if ((t & 31) == 0) producer_role(p, ms, smem);
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if ((t & 31) == 0) mma_role(p, ms, smem);
    __syncwarp();
  } else if (tq8(p)) {
    dequant_role(p, ms, smem);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(ms.tmem_base, kTmemCols);
}

// ----------------------------------------------------------------- host
size_t al256(size_t b) { return (b + 255) & ~size_t(255); }

// This build's dynamic shared memory (the two kernels' maps differ).
constexpr size_t kernel_smem_bytes() { return kOffMisc + sizeof(Misc) + 1024; }
static_assert(kernel_smem_bytes() <= 232448, "more shared memory than a CTA may have");

struct SyncLayout {
  size_t tile_cnt, ready, ss_cnt, ss, rexp, head_done, codepk, decided, abort_flag;
  size_t zeroed;   // bytes from the start zeroed before each launch
  size_t ss_part;  // deterministic mode's partial sums (written before they are read; not zeroed)
  size_t total;
  int NCH, MT, KS, NGEMM;
};

SyncLayout sync_layout(const qp_geometry& g, int B) {
  SyncLayout S{};
  const size_t R1 = size_t(2) * B;
  S.NCH = int(R1 <= size_t(kMaxNc) ? 1 : (R1 + kMaxNc - 1) / kMaxNc);
  const int qkvw = (g.n_q_heads + 2 * g.n_kv_heads) * 128;
  int mt = g.hidden;
  if (qkvw > mt) mt = qkvw;
  if (2 * g.ffn > mt) mt = 2 * g.ffn;
  if (g.vocab > mt) mt = g.vocab;
  S.MT = mt / kTileM;
  int ks = g.hidden;
  if (g.talker_hidden > ks) ks = g.talker_hidden;
  if (g.n_q_heads * 128 > ks) ks = g.n_q_heads * 128;
  if (g.ffn > ks) ks = g.ffn;
  S.KS = ks / kKs;
  S.NGEMM = 1 + g.n_steps * (4 * g.layers + 1) + (g.code_embed_dim != g.hidden) * (g.n_steps - 1);
  size_t o = 0;
  S.tile_cnt = o; o += al256(size_t(S.NGEMM) * S.NCH * S.MT * 4);
  S.ready = o;    o += al256(size_t(S.NGEMM) * S.NCH * S.KS * 4);
  S.ss_cnt = o;   o += al256(size_t(S.NGEMM) * S.NCH * 4);
  S.ss = o;       o += al256(size_t(S.NGEMM) * R1 * 4);
  S.rexp = o;     o += al256(size_t(S.NGEMM) * R1 * 4);
  S.head_done = o; o += al256(size_t(g.n_steps) * S.NCH * 4);
  S.codepk = o;   o += al256(size_t(g.n_steps) * B * 8);
  S.decided = o;  o += al256(size_t(g.n_steps) * B * 4);
  S.abort_flag = o; o += 256;
  S.zeroed = o;
  S.ss_part = o;  o += al256(size_t(S.NGEMM) * (g.hidden / kTileM) * R1 * 4);
  S.total = o;
  return S;
}

void fill_params(PParams& p, const qp_handle* h, const RunArgs& a, uint8_t* scratch, const Scratch& L,
                 uint8_t* sync, const SyncLayout& S, int bmax) {
  const qp_geometry& g = h->g;
  p.d = g.hidden; p.qw = g.n_q_heads * 128; p.kvw = g.n_kv_heads * 128; p.F = g.ffn; p.V = g.vocab;
  p.th = g.talker_hidden; p.L = g.layers; p.n_q = g.n_q_heads; p.n_kv = g.n_kv_heads; p.n_steps = g.n_steps;
  p.q0_vocab = g.q0_vocab; p.eps = g.rms_eps; p.q8 = h->wfmt == WF_Q8_0; p.q8_head = h->hfmt == WF_Q8_0;
  p.embed_f16 = h->embed_f16;
  p.proj_in = g.code_embed_dim != g.hidden;
  p.w_proj = h->proj.w; p.s_proj = h->proj.scale; p.b_proj = h->b_proj; p.e0 = h->e0;
  for (int l = 0; l < g.layers; ++l) {
    const LayerW& Lw = h->layer[l];
    const PackedMat* m[4] = {&Lw.qkv, &Lw.o, &Lw.gu, &Lw.down};
    for (int i = 0; i < 4; ++i) { p.layer[l].w[i] = m[i]->w; p.layer[l].s[i] = m[i]->scale; }
    p.layer[l].attn_norm = Lw.attn_norm; p.layer[l].q_norm = Lw.q_norm;
    p.layer[l].k_norm = Lw.k_norm; p.layer[l].ffn_norm = Lw.ffn_norm;
  }
  p.out_norm = h->out_norm;
  for (int j = 0; j < g.n_steps; ++j) {
    p.embed[j] = h->embed[j]; p.embed_ss[j] = h->embed_ss[j];
    p.w_head[j] = h->head[j].w; p.s_head[j] = h->head[j].scale;
  }
  p.rope_cs = h->rope_cs;
  p.x1 = reinterpret_cast<float*>(scratch + L.x1);
  p.xk = reinterpret_cast<float*>(scratch + L.xk);
  for (int i = 0; i < 5; ++i) p.a1[i] = reinterpret_cast<uint16_t*>(scratch + L.a1[i]);
  for (int i = 0; i < 4; ++i) p.ak[i] = reinterpret_cast<uint16_t*>(scratch + L.ak[i]);
  p.ahead = reinterpret_cast<uint16_t*>(scratch + L.ahead);
  p.acc1_qkv = reinterpret_cast<float*>(scratch + L.acc1_qkv);
  p.acck_qkv = reinterpret_cast<float*>(scratch + L.acck_qkv);
  p.acc1_gu = reinterpret_cast<float*>(scratch + L.acc1_gu);
  p.acck_gu = reinterpret_cast<float*>(scratch + L.acck_gu);
  p.logits = reinterpret_cast<float*>(scratch + L.logits);
  p.kv = reinterpret_cast<uint16_t*>(scratch + L.kv);
  p.Bmax = bmax;
  p.tile_cnt = reinterpret_cast<unsigned*>(sync + S.tile_cnt);
  p.ready = reinterpret_cast<unsigned*>(sync + S.ready);
  p.ss_cnt = reinterpret_cast<unsigned*>(sync + S.ss_cnt);
  p.ss = reinterpret_cast<float*>(sync + S.ss);
  p.rexp = reinterpret_cast<int*>(sync + S.rexp);
  p.head_done = reinterpret_cast<unsigned*>(sync + S.head_done);
  p.codepk = reinterpret_cast<unsigned long long*>(sync + S.codepk);
  p.decided = reinterpret_cast<unsigned*>(sync + S.decided);
  p.abort_flag = reinterpret_cast<int*>(sync + S.abort_flag);
  p.status = h->status;
  p.spin_limit = h->wait_ticks > 0 ? h->wait_ticks : kSpinLimit;
  p.withhold = h->withhold_gemm;
  p.det = h->deterministic ? 1 : 0;
  p.ss_part = reinterpret_cast<float*>(sync + S.ss_part);
  p.NCH = S.NCH; p.MT = S.MT; p.KS = S.KS; p.NGEMM = S.NGEMM;
  p.trace = h->trace; p.trace_n = h->trace_phases;
  p.B = a.B; p.H = a.H; p.q0 = a.q0; p.out_codes = a.out_codes; p.out_logits = a.out_logits; p.forced = a.forced;
  p.temperature = a.temperature; p.top_k = a.top_k; p.gumbel = a.gumbel;
}

// Zero what must start at zero, then launch.
qp_status launch(qp_handle* h, PParams& p, uint8_t* scratch, const Scratch& L, uint8_t* sync, const SyncLayout& S,
                 cudaStream_t s, std::atomic<bool>* attr_done) {
  const qp_geometry& g = h->g;
  if (!attr_done->load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(TILE_KERNEL, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kernel_smem_bytes())) != cudaSuccess) {
      cudaGetLastError();
      return QP_ERR_CUDA;
    }
    attr_done->store(true, std::memory_order_release);
  }
  const size_t B = size_t(p.B), qkvw = size_t(g.n_q_heads + 2 * g.n_kv_heads) * 128, F2 = size_t(2) * g.ffn;
  cudaError_t e = cudaMemsetAsync(sync, 0, S.zeroed, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(scratch + L.acc1_qkv, 0, 2 * B * qkvw * 4, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(scratch + L.acck_qkv, 0, B * qkvw * 4, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(scratch + L.acc1_gu, 0, 2 * B * F2 * 4, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(scratch + L.acck_gu, 0, B * F2 * 4, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(scratch + L.logits, 0, B * size_t(g.vocab) * 4, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return QP_ERR_CUDA;
  }
  void* args[] = {&p};
  if (cudaLaunchCooperativeKernel(reinterpret_cast<void*>(TILE_KERNEL), dim3(h->num_sms), dim3(kThreads), args,
                                  kernel_smem_bytes(), s) != cudaSuccess) {
    cudaGetLastError();
    return QP_ERR_CUDA;
  }
  return QP_OK;
}

// Per device: the kernel's shared-memory limit has been set.  First calls
// from several host threads may race to set it (an idempotent call); the
// flag itself is atomic.
std::atomic<bool> g_attr_done[64];

}  // namespace

#if QP_TILE_Q8

// The Q8_0 kernel's launch; run_frames_persistent and run_frames_static
// (16-bit build) send calls with Q8_0 matrices here.
qp_status run_tile_q8(qp_handle* h, const RunArgs& a, uint8_t* scratch, const Scratch& L, int bmax, cudaStream_t s) {
  const SyncLayout S = sync_layout(h->g, a.B);
  PParams p{};
  fill_params(p, h, a, scratch, L, scratch + L.sync, S, bmax);
  std::atomic<bool>* done = h->device >= 0 && h->device < 64 ? &g_attr_done[h->device] : nullptr;
  std::atomic<bool> local(false);
  return launch(h, p, scratch, L, scratch + L.sync, S, s, done ? done : &local);
}

#else

size_t persistent_smem_bytes() { return kernel_smem_bytes(); }

Scratch scratch_layout(const qp_geometry& g, int bmax) {
  Scratch L{};
  const size_t R1 = size_t(2) * bmax, RK = size_t(bmax), o1 = operand_rows(R1), ok = operand_rows(RK);
  const size_t d = g.hidden, qw = size_t(g.n_q_heads) * 128, kvw = size_t(g.n_kv_heads) * 128, F = g.ffn;
  const size_t qkvw = qw + 2 * kvw, th = g.talker_hidden, V = g.vocab;
  size_t o = 0;
  L.x1 = o; o += al256(R1 * d * 4);
  L.xk = o; o += al256(RK * d * 4);
  const size_t k1[5] = {th, d, qw, d, F};
  for (int i = 0; i < 5; ++i) { L.a1[i] = o; o += al256(o1 * k1[i] * 2); }
  const size_t kk[4] = {d, qw, d, F};
  for (int i = 0; i < 4; ++i) { L.ak[i] = o; o += al256(ok * kk[i] * 2); }
  L.ahead = o; o += al256(ok * d * 2);
  L.acc1_qkv = o; o += al256(R1 * qkvw * 4);
  L.acck_qkv = o; o += al256(RK * qkvw * 4);
  L.acc1_gu = o;  o += al256(R1 * 2 * F * 4);
  L.acck_gu = o;  o += al256(RK * 2 * F * 4);
  L.logits = o;   o += al256(RK * V * 4);
  L.acc_qkv_b = o; o += al256(R1 * qkvw * 4);
  L.kv = o;       o += al256(size_t(g.layers) * RK * (g.n_steps + 1) * 2 * kvw * 2);
  L.sync = o;
  L.total = o + sync_layout(g, bmax).total;
  return L;
}

size_t sync_bytes(const qp_geometry& g, int B) { return sync_layout(g, B).total; }

qp_status run_frames_persistent(qp_handle* h, const RunArgs& a, cudaStream_t s) {
  if (a.temperature > 0.f && h->g.vocab > kMaxVocab) return QP_ERR_ARG;
  uint8_t* scratch = static_cast<uint8_t*>(h->sarena);
  if (h->wfmt == WF_Q8_0) return run_tile_q8(h, a, scratch, h->scr, h->max_batch, s);
  const SyncLayout S = sync_layout(h->g, a.B);
  PParams p{};
  fill_params(p, h, a, scratch, h->scr, scratch + h->scr.sync, S, h->max_batch);
  std::atomic<bool>* done = h->device >= 0 && h->device < 64 ? &g_attr_done[h->device] : nullptr;
  std::atomic<bool> local(false);
  return launch(h, p, scratch, h->scr, scratch + h->scr.sync, S, s, done ? done : &local);
}

// ---------------------------------------------------------------------------
// Allocation-free entry point.
//
// Callers whose device memory is owned by someone else cannot have this
// library call cudaMalloc on their behalf: a process whose framework
// allocator has already reserved the GPU's memory, or a real-time audio path
// that forbids allocation once it is running.  qp_predict_frames_static
// runs the same kernel as qp_predict_frames, but its scratch (residual
// streams, operands, accumulators, logits, KV cache and synchronisation
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
// Per device, looked up on the first call (atomic: first calls from several
// host threads may race; each stores the same address).
std::atomic<void*> g_static_ptr[kMaxDevices];
std::atomic<bool> g_static_attr[kMaxDevices];
}  // namespace

qp_status run_frames_static(qp_handle* h, const RunArgs& a, cudaStream_t s) {
  const qp_geometry& g = h->g;
  if (a.B < 1 || a.B > kStaticMaxFrames) return QP_ERR_ARG;
  const Scratch L = scratch_layout(g, a.B);
  if (L.total > kStaticScratchBytes) return QP_ERR_ARG;
  if (h->device < 0 || h->device >= kMaxDevices) return QP_ERR_ARG;
  // once per device, with that device current: the array's device address
  if (!g_static_ptr[h->device].load(std::memory_order_acquire)) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return QP_ERR_CUDA;
    }
    g_static_ptr[h->device].store(ptr, std::memory_order_release);
  }
  uint8_t* base = static_cast<uint8_t*>(g_static_ptr[h->device].load(std::memory_order_acquire));
  const SyncLayout S = sync_layout(g, a.B);
  RunArgs ga = a;
  ga.forced = nullptr;
  ga.temperature = 0.f; ga.top_k = 0; ga.gumbel = nullptr;
  const bool sm = small_supported(h, ga);
  if (h->engine == QP_ENGINE_SMALL && !sm) return QP_ERR_ARG;
  const bool pick = h->engine == QP_ENGINE_SMALL || (h->engine == QP_ENGINE_AUTO && a.B <= kSmallAutoFrames);
  if (h->deterministic && h->engine == QP_ENGINE_SMALL) return QP_ERR_ARG;   // the tile engine serves that mode
  if (sm && pick && !h->deterministic) return run_frames_small(h, ga, base, L, a.B, s);
  if (h->wfmt == WF_Q8_0) return run_tile_q8(h, ga, base, L, a.B, s);
  PParams p{};
  fill_params(p, h, ga, base, L, base + L.sync, S, a.B);
  // the launch zeroes the synchronisation words and accumulators; every
  // other byte is written before it is read within the call
  return launch(h, p, base, L, base + L.sync, S, s, &g_static_attr[h->device]);
}

#endif

}  // namespace qp
