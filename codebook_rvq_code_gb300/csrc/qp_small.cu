// The Code Predictor frame loop for small batches (at most 64 frames): one
// persistent kernel, scheduled for latency.
//
// It computes what qp_persistent.cu computes (the whole frame loop as one
// fixed GPU program over a preallocated KV cache: "テキスト音声合成モデルを50
// ミリ秒未満で応答させる方法", section "Qwen3-TTSの最適化方法", item 3).  The
// contractions use the same tensor-core shape -- 128 weight rows on M, the
// activation rows on N (16..128), f16 operands, f32 accumulators in TMEM --
// and K is split across the SMs in 128-column slices so that every SM streams
// an equal share of each weight matrix.  What differs is how a dependent step
// completes:
//
//   * each (128-row tile, K slice) unit adds its f32 partial product straight
//     into the destination (the residual stream for projection, O and down;
//     the q|k|v, gate|up and logit accumulators otherwise) and counts itself
//     done; a GEMM waits for one counter to reach the previous GEMM's unit
//     count.  There is no finishing pass over a completed tile;
//   * the consumer warps of the CTA that runs a unit build its operand slice
//     in shared memory from those f32 sources: x * w_norm, silu(g) * u, the
//     f16 conversion -- the work the tile engine's finishing pass does once;
//   * the rows' RMS scale is applied where a complete residual row is at
//     hand: the gate/up GEMM (and step 1's head) computes it from the rows
//     and scales its partials before they are added; the QKV GEMM adds
//     unscaled partials and each attention item scales its frame's q, k and
//     v; from step 2 the head adds unscaled logits and the decision scales
//     the row it copies out.
//
// Roles per CTA (one CTA per SM): warps 0-7 consume (operand builds,
// accumulator drains, attention, step inputs, decisions), warp 8 streams
// weights, warp 9 issues the MMAs.  Every wait is bounded and honours a
// grid-wide abort flag; each role walks the program in one order and waits
// only on work earlier in that order, and all CTAs are co-resident
// (cooperative launch).
#include <algorithm>
#include <atomic>

#include "qp_device.cuh"

namespace qp {

namespace {

constexpr int kSmConsumerWarps = 8;
constexpr int kSmConsumers = kSmConsumerWarps * 32;
constexpr int kSmProducerWarp = 8;
constexpr int kSmMmaWarp = 9;
constexpr int kSmThreads = 10 * 32;

constexpr uint32_t kSmWSlot = kTileM * kKs * 2;      // one 128 x 128 f16 weight slice
constexpr int kSmNW = 4;                             // weight ring slots
constexpr uint32_t kSmOpBytes = 65536;               // operand slices, 128 K x N rows f16 each
constexpr int kSmMaxOp = 8;
constexpr uint32_t kSmOffW = 0;
constexpr uint32_t kSmOffOp = kSmNW * kSmWSlot;
constexpr uint32_t kSmOffKeys = kSmOffOp + kSmOpBytes;   // top-k keys, or the drain's transpose buffer
constexpr uint32_t kSmOffMisc = kSmOffKeys + kMaxVocab * 4;
constexpr uint32_t kSmTmemCols = 256;                // two accumulators of up to 128 columns

enum { SBAR_CONS = 1, SBAR_HALF0 = 2 };   // SBAR_HALF0 + h: consumer half h (4 warps)
enum { S_PROJ = 0, S_QKV, S_O, S_GU, S_DOWN, S_HEAD };
// The QKV projection without the row scale (a code path of the S_QKV GEMM):
// each attention item scales its frame's q, k and v itself, so the GEMM
// needs no row-scale pass.
constexpr int S_QKVU = 7;

// Call modes: a whole frame loop; step 1 only, into state slots; one step
// of rows at mixed steps, from state slots (include/qp_sched.h).
enum { SM_RUN = 0, SM_BEGIN = 1, SM_STEP = 2 };
// This translation unit's kernel: the greedy frame loop (SM_RUN); built from
// qp_small_sampled.cu, the frame loop with Gumbel top-k sampling; built from
// qp_small_slots.cu, the state-slot calls (SM_BEGIN, SM_STEP, greedy).  The
// builds keep each kernel free of the others' code and registers: the
// kernel carries every section inline, and code it does not run still costs
// registers and instruction fetch.
#ifndef QP_SMALL_SLOTS
#define QP_SMALL_SLOTS 0
#endif
#ifndef QP_SMALL_SAMPLED
#define QP_SMALL_SAMPLED 0
#endif
constexpr bool kSmSlots = QP_SMALL_SLOTS != 0;
constexpr bool kSmSampled = QP_SMALL_SAMPLED != 0;

struct SMisc {
  uint64_t wfull[kSmNW], wempty[kSmNW];
  uint64_t ofull[kSmMaxOp], oempty[kSmMaxOp];
  uint64_t accfull[2], accempty[2];
  uint64_t mmadone;
  uint32_t tmem_base;
  int flag[4];
  int fail;
  unsigned evc;
  unsigned long long redu[kSmConsumerWarps];
  int sel[2];
  int hist[256];
  TopkScratch topk[2];   // sampling: one frame per consumer half
  int hflag[2];
  float inv[kMaxNc];
  float ssp[kSmConsumerWarps][kMaxNc];   // per-warp partial sums of squares
  int bcast;
  uint32_t ouse[kSmMaxOp];   // consumers (thread 0): fills of each operand slot so far
  uint32_t ouse_m[kSmMaxOp]; // MMA thread: fills of each operand slot consumed so far
};

struct SLayer {
  const uint16_t* w[4];    // qkv, o, gu, down: tile-packed f16 (qp_weights.cu); for Q8_0 matrices the hi image
  const uint16_t* wl[4];   // Q8_0 matrices: the lo image (hi + lo = d * q), else null
  const float* attn_norm; const float* q_norm; const float* k_norm; const float* ffn_norm;
};

struct SParams {
  int d, qw, kvw, F, V, th, L, n_q, n_kv, n_steps, q0_vocab;
  float eps;
  const uint16_t* w_proj; const uint16_t* w_proj_lo; const float* b_proj; const uint16_t* e0;
  SLayer layer[kMaxLayers];
  const float* out_norm;
  const uint16_t* embed[kMaxSteps];
  const uint16_t* w_head[kMaxSteps];
  const uint16_t* w_head_lo[kMaxSteps];   // Q8_0 heads: the lo images, else null
  const float2* rope_cs;
  // scratch (rows: 2B at step 1, B later)
  float* x;                // residual stream [row][d]
  uint16_t* a_o;           // attention output, f16 [row][q_width]
  float* acc_qkv[2];       // [row][q_width + 2 kv_width], unscaled (attention applies the row's 1/RMS); layers alternate
  float* acc_gu;           // [row][2 ffn]: gate then up, scaled by the row's RMS
  float* logits;           // [frame][vocab]
  uint16_t* kv;            // f16 [layer][frame][pos][k|v][kv_width]
  int Bmax;                // frame stride of the KV cache
  // per-call synchronisation (zeroed before the launch)
  unsigned* done;          // [gemm]: units finished
  unsigned* qkv_tile;      // [step][layer][128-row tile of q|k|v]: K slices finished
  unsigned* att;           // [step][layer]: attention items finished
  unsigned* prep;          // [step]: input rows finished
  unsigned* decided;       // [step][frame]: sampled code + 1
  int* rexp;               // [gemm][row]: range exponent e of the operand row (f16(v * 2^-e); 0 = unscaled)
  int* abort_flag; int* status;
  long long spin_limit;    // clock64 ticks a wait may take before the call aborts
  int withhold;            // testing (qp_debug.h): GEMM whose count CTA run 0 skips; -1 none
  int NGEMM, NHT;
  unsigned long long* trace; int trace_n;
  // the call
  int proj_in;             // code tables are Talker-wide: each step's input passes through small_to_mtp
  bool embed_f16;          // embedding tables are f16, else bf16
  // state-slot calls (SM_BEGIN, SM_STEP); rows of an SM_STEP call are sorted
  // by step, and row b is the caller's row row_perm[b]
  int mode, n_run, k_first;        // steps run this call: k_first .. k_first + n_run - 1
  int n_groups, group_rows;        // SM_STEP: step groups, rows of the largest
  // row b's KV state slot, step and caller row; rows [group_start[h],
  // group_start[h + 1]) are at step group_step[h] (SM_STEP)
  int32_t row_slot[kSmallMaxFrames], row_step[kSmallMaxFrames], row_perm[kSmallMaxFrames];
  int32_t group_start[kMaxSteps + 1], group_step[kMaxSteps];
  const int32_t* code_in;          // SM_STEP: device [B], caller order
  int32_t* in_code;        // [step][frame]: the code whose embedding is step k's input (proj_in)
  int B; const float* H; const int32_t* q0; int32_t* out_codes; float* out_logits; const int32_t* forced;
  float temperature; int top_k; const float* gumbel;
};

__device__ __forceinline__ int sm_mode(const SParams& p) { return kSmSlots ? p.mode : int(SM_RUN); }
__device__ __forceinline__ int sm_k_first(const SParams& p) { return kSmSlots ? p.k_first : 1; }
__device__ __forceinline__ int sm_n_run(const SParams& p) { return kSmSlots ? p.n_run : p.n_steps; }
__device__ __forceinline__ bool sm_sampled(const SParams& p) { return kSmSampled && p.temperature > 0.f; }

// One GEMM of the program: n_mt tiles of 128 weight rows x n_ks slices of K.
struct SG {
  int kind, k, l, R, N, n_mt, n_ks, ld;
  int r0;   // first activation / output row (a step group's head)
  bool scaled;
  const uint16_t* w; float* out;
  const uint16_t* wl;   // the lo image of a Q8_0 matrix (a unit then multiplies two slices), else null
};
// The program: GEMM 0 is step 1's projection (rows H_b, E0[q0_b]); step k
// then has, with Talker-wide code tables and k >= 2, the projection of its
// input rows, then 4 GEMMs per layer (QKV, O, GU, down) and the head.
__device__ __forceinline__ int sgi_base(const SParams& p, int k) {
  // an SM_STEP call's program: [projection], 4 GEMMs per layer, one head per step group
  if (sm_mode(p) == SM_STEP) return p.proj_in;
  return 1 + (k - 1) * (4 * p.L + 1) + p.proj_in * (k - 1);
}
__device__ __forceinline__ int sgi_of(const SParams& p, int k, int l, int t) { return sgi_base(p, k) + 4 * l + t; }
__device__ __forceinline__ int sgi_head(const SParams& p, int k) { return sgi_base(p, k) + 4 * p.L; }
__device__ __forceinline__ int sgi_proj(const SParams& p, int k) { return k == 1 ? 0 : sgi_base(p, k) - 1; }
// the KV state of activation row b's frame: its slot in state-slot calls
__device__ __forceinline__ int sm_slot(const SParams& p, int b) { return sm_mode(p) == SM_RUN ? b : p.row_slot[b]; }
__device__ __forceinline__ int sm_cols(int R) { return (R + 15) & ~15; }

__device__ SG sgemm(const SParams& p, int gi) {
  SG g;
  g.scaled = false;
  g.r0 = 0;
  int r = -1;   // the GEMM's place in its step: -1 the projection, 4L the head
  if (sm_mode(p) == SM_STEP) {
    g.k = 2;
    r = gi - p.proj_in;
    if (r == 4 * p.L) {   // every step group's head: tile mt is group mt / (V / 128)'s
      g.kind = S_HEAD; g.l = p.L - 1; g.R = p.group_rows; g.n_mt = p.n_groups * (p.V / kTileM);
      g.n_ks = p.d / kKs; g.w = nullptr; g.wl = p.w_head_lo[0]; g.out = p.logits; g.ld = p.V;
      g.N = sm_cols(g.R);
      return g;
    }
  } else if (gi == 0) {
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
  g.R = g.k == 1 ? 2 * p.B : p.B;
  if (r < 0) {
    g.kind = S_PROJ; g.l = 0; g.n_mt = p.d / kTileM; g.n_ks = p.th / kKs;
    g.w = p.w_proj; g.wl = p.w_proj_lo; g.out = p.x; g.ld = p.d;
  } else {
    if (r == 4 * p.L) {
      g.kind = S_HEAD; g.l = p.L - 1; g.R = p.B; g.n_mt = p.V / kTileM; g.n_ks = p.d / kKs;
      g.w = p.w_head[g.k - 1]; g.wl = p.w_head_lo[g.k - 1]; g.out = p.logits; g.ld = p.V; g.scaled = true;
    } else {
      g.l = r / 4;
      const SLayer& L = p.layer[g.l];
      g.wl = L.wl[r % 4];
      switch (r % 4) {
        case 0: g.kind = S_QKV; g.n_mt = (p.qw + 2 * p.kvw) / kTileM; g.n_ks = p.d / kKs; g.w = L.w[0];
                g.out = p.acc_qkv[((g.k - 1) * p.L + g.l) & 1]; g.ld = p.qw + 2 * p.kvw; g.scaled = true; break;
        case 1: g.kind = S_O; g.n_mt = p.d / kTileM; g.n_ks = p.qw / kKs; g.w = L.w[1]; g.out = p.x; g.ld = p.d; break;
        case 2: g.kind = S_GU; g.n_mt = 2 * p.F / kTileM; g.n_ks = p.d / kKs; g.w = L.w[2];
                g.out = p.acc_gu; g.ld = 2 * p.F; g.scaled = true; break;
        default: g.kind = S_DOWN; g.n_mt = p.d / kTileM; g.n_ks = p.F / kKs; g.w = L.w[3]; g.out = p.x; g.ld = p.d; break;
      }
    }
  }
  g.N = sm_cols(g.R);
  return g;
}

// The activation rows [r0, r0 + R) of tile mt, and the weight slice of unit
// s.  An SM_STEP call's head GEMM holds one head per step group, each with
// its own rows and matrix.
__device__ __forceinline__ bool sm_grouped(const SParams& p, const SG& g) {
  return kSmSlots && g.kind == S_HEAD && sm_mode(p) == SM_STEP;
}
__device__ __forceinline__ void sm_rows(const SParams& p, const SG& g, int mt, int& r0, int& R) {
  if (sm_grouped(p, g)) {
    const int h = mt / (p.V / kTileM);
    r0 = p.group_start[h];
    R = p.group_start[h + 1] - r0;
  } else {
    r0 = g.r0;
    R = g.R;
  }
}
// Image 0 is the 16-bit matrix (or a Q8_0 matrix's hi image), image 1 a
// Q8_0 matrix's lo image.
__device__ __forceinline__ const uint8_t* sm_slice(const SParams& p, const SG& g, int s, int img = 0) {
  if (sm_grouped(p, g)) {
    const int per = (p.V / kTileM) * g.n_ks, h = s / per;
    const uint16_t* m = img ? p.w_head_lo[p.group_step[h] - 1] : p.w_head[p.group_step[h] - 1];
    return reinterpret_cast<const uint8_t*>(m) + size_t(s - h * per) * kSmWSlot;
  }
  return reinterpret_cast<const uint8_t*>(img ? g.wl : g.w) + size_t(s) * kSmWSlot;
}

// GEMMs whose partials are scaled by the input row's 1/RMS.  From step 2 on
// the head's logits are added unscaled: a positive row scale does not move
// the argmax, and the frame's decision applies it where values are copied
// out or sampled, from the frame's residual row, which only that decision's
// CTA overwrites afterwards.  (At step 1 the head's rows are 2b+1, which the
// next step's inputs overwrite from other CTAs, so there the GEMM scales.)
template <int KIND>
constexpr bool kScaled = KIND == S_QKV || KIND == S_GU;
template <int KIND>
__device__ __forceinline__ bool sm_scaled(const SG& g) { return kScaled<KIND> || (KIND == S_HEAD && g.k == 1); }
template <int KIND>
constexpr bool kQkv = KIND == S_QKV || KIND == S_QKVU;
// GEMMs whose operand rows come from the residual stream or from H: each
// row is built as f16(v * 2^-e) (qp_device.cuh, range_exp), and 2^e is
// applied with the row scale where that is applied: to the partial products
// of the gate/up GEMM, step 1's head and step 1's projection as they are
// added; by the attention items (QKV) and by the decision (the head from
// step 2), which read the accumulated values.
template <int KIND>
constexpr bool kRange = KIND == S_PROJ || kQkv<KIND> || KIND == S_GU || KIND == S_HEAD;
__device__ __forceinline__ int* sm_rexp(const SParams& p, int gi, int row) { return p.rexp + size_t(gi) * 2 * p.B + row; }

// The operand ring of a GEMM: slots of N x 128 f16 (the GEMM's own width),
// as many as fit the region.  A CTA's unit i of the GEMM uses slot i % n.
__device__ __forceinline__ uint32_t sm_op_bytes(const SG& g) { return uint32_t(g.N) * kKs * 2; }
__device__ __forceinline__ uint32_t sm_op_slots(const SG& g) {
  const uint32_t n = kSmOpBytes / sm_op_bytes(g);
  return n < uint32_t(kSmMaxOp) ? n : uint32_t(kSmMaxOp);
}

// This CTA's contiguous run [beg, end) of a GEMM's units, ordered (tile, K
// slice); the runs rotate with the GEMM index so that the CTAs with the
// larger share change from one GEMM to the next.
__device__ __forceinline__ void sm_run(const SG& g, int gi, int& beg, int& end) {
  const int G = gridDim.x, c = int((unsigned(blockIdx.x) + unsigned(gi) * 37u) % unsigned(G));
  const int total = g.n_mt * g.n_ks;
  beg = int((long long)total * c / G);
  end = int((long long)total * (c + 1) / G);
}

// sync-region accessors
__device__ __forceinline__ unsigned* sm_done(const SParams& p, int gi) { return p.done + gi; }
__device__ __forceinline__ unsigned* sm_qkv_tile(const SParams& p, int k, int l, int t) {
  return p.qkv_tile + (size_t(k - 1) * p.L + l) * p.NHT + t;
}
__device__ __forceinline__ unsigned* sm_att(const SParams& p, int k, int l) { return p.att + (k - 1) * p.L + l; }
__device__ __forceinline__ unsigned* sm_prep(const SParams& p, int k) { return p.prep + (k - 1); }

// The counter a GEMM's operand depends on and the value that completes it.
__device__ void sm_ready(const SParams& p, int gi, const unsigned*& ctr, unsigned& want) {
  const SG g = sgemm(p, gi);
  auto all_of = [&](int gp) { const SG q = sgemm(p, gp); ctr = sm_done(p, gp); want = unsigned(q.n_mt * q.n_ks); };
  switch (g.kind) {
    case S_PROJ: ctr = sm_prep(p, g.k); want = unsigned(g.R); return;   // the step's input rows
    case S_QKV:
      if (g.l > 0 || (g.k > 1 && p.proj_in)) { all_of(gi - 1); return; }   // previous down, or the projection
      if (g.k == 1) { all_of(0); return; }              // the input projection
      ctr = sm_prep(p, g.k); want = unsigned(p.B); return;   // the step's input rows
    case S_O: ctr = sm_att(p, g.k, g.l); want = unsigned(p.B * p.n_kv); return;
    default: all_of(gi - 1); return;                     // GU: O; DOWN: GU; HEAD: the last DOWN
  }
}

// ------------------------------------------------------------ tracing
// Section stamps [section][cta][start, end], then a per-CTA event log:
// consumer events in [0, 8192), MMA-warp events in [8192, 16384); one word =
// (globaltimer ns mod 2^48) << 16 | code << 12 | gemm.
enum {
  SEV_READY = 1, SEV_BUILT = 2, SEV_COMMIT = 3,   // consumers: readiness seen, operands built; MMA: segment committed
  SEV_ACC = 4, SEV_PUBLISHED = 6,                 // consumers: accumulator seen, units released
  SEV_ATT_READY = 8, SEV_ATT_DONE = 9,            // attention warp, per item
  SEV_WEIGHTS = 10, SEV_ISSUE = 11,               // MMA: waited for a weight slice; producer: copy issued
  SEV_WEIGHTS_READY = 12                          // MMA: the weight slice was already there
};
__device__ __forceinline__ unsigned long long* sm_ev_base(const SParams& p) {
  return p.trace ? p.trace + size_t(p.trace_n) * gridDim.x * 2 + size_t(blockIdx.x) * 16384 : nullptr;
}
__device__ __forceinline__ unsigned long long sm_ev_word(int code, int gi) {
  return ((globaltimer_ns() & 0xFFFFFFFFFFFFull) << 16) | (unsigned long long)(code & 15) << 12 | unsigned(gi & 4095);
}
// Compiled in only with QP_TRACE (qp_debug.h): the hooks sit on the loop's
// critical path, where even untaken branches cost instruction fetch.
#ifdef QP_TRACE
__device__ __forceinline__ void sm_ev_mma(const SParams& p, unsigned& idx, int code, int gi) {
  unsigned long long* b = sm_ev_base(p);
  if (b && idx < 8192) b[8192 + idx++] = sm_ev_word(code, gi);
}
__device__ __forceinline__ void sm_ev(const SParams& p, unsigned* cnt, int code, int gi) {
  unsigned long long* b = sm_ev_base(p);
  if (b) {
    const unsigned i = atomicAdd(cnt, 1u);
    if (i < 8192) b[i] = sm_ev_word(code, gi);
  }
}
__device__ __forceinline__ void sm_trace_mark(const SParams& p, int sec, int which) {
  if (p.trace && threadIdx.x == 0 && sec < p.trace_n)
    p.trace[(size_t(sec) * gridDim.x + blockIdx.x) * 2 + which] = globaltimer_ns();
}
#else
__device__ __forceinline__ void sm_ev_mma(const SParams&, unsigned&, int, int) {}
__device__ __forceinline__ void sm_ev(const SParams&, unsigned*, int, int) {}
__device__ __forceinline__ void sm_trace_mark(const SParams&, int, int) {}
#endif

// ---------------------------------------------------------------- producer
// Streams the weight slices of this CTA's units, in program order, through
// the ring; it depends on nothing, so it runs ahead by the ring's depth.
__device__ void sm_producer(const SParams& p, SMisc& ms, uint8_t* smem) {
  const uint64_t pol = policy_evict_first();
  uint32_t it = 0;
  for (int gi = 0; gi < p.NGEMM; ++gi) {
    const SG g = sgemm(p, gi);
    int beg, end;
    sm_run(g, gi, beg, end);
    const int nimg = g.wl ? 2 : 1;   // a Q8_0 matrix's unit takes its hi and lo slices
    for (int s = beg; s < end; ++s) {
      for (int img = 0; img < nimg; ++img) {
        const uint32_t slot = it % kSmNW, u = it / kSmNW;
        if (u > 0 && !mwait(p, &ms.wempty[slot], (u - 1) & 1)) goto drain;
        sm_ev(p, &ms.evc, SEV_ISSUE, gi);
        mbar_expect_tx(&ms.wfull[slot], kSmWSlot);
        // tile mt, slice ks of the tile-packed matrix: one contiguous 32 KB run
        bulk_g2s_stream(smem + kSmOffW + slot * kSmWSlot, sm_slice(p, g, s, img), kSmWSlot, &ms.wfull[slot], pol);
        ++it;
      }
    }
  }
drain:
  for (uint32_t k = it > uint32_t(kSmNW) ? it - kSmNW : 0; k < it; ++k) mbar_wait(&ms.wfull[k % kSmNW], (k / kSmNW) & 1);
}

// --------------------------------------------------------------- MMA warp
// Per unit: the weight slice (A, 128 rows) and the operand slice the
// consumers built (B, N rows), 8 MMAs of K = 16 into the accumulator of the
// unit's segment (a run of consecutive K slices of one tile).
__device__ void sm_mma(const SParams& p, SMisc& ms, uint8_t* smem) {
  uint32_t wit = 0, seg = 0;
  uint32_t* ouse = ms.ouse_m;
  unsigned evi = 0;
  for (int gi = 0; gi < p.NGEMM; ++gi) {
    const SG g = sgemm(p, gi);
    int beg, end;
    sm_run(g, gi, beg, end);
    const uint32_t idesc = idesc_f16(kTileM, g.N);
    const uint32_t blb = uint32_t(g.N / 8) * 128;   // operand K-direction core-matrix stride
    const uint32_t nop = sm_op_slots(g), obytes = sm_op_bytes(g);
    const uint32_t nimg = g.wl ? 2u : 1u;   // Q8_0: the hi and lo slices, multiplied into one accumulator
    for (int s = beg; s < end; ++s) {
      const int ks = s % g.n_ks;
      const bool first = s == beg || ks == 0;
      const bool last = s == end - 1 || ks == g.n_ks - 1;
      const uint32_t ws = wit % kSmNW, os = uint32_t(s - beg) % nop, tb = seg & 1;
      if (mbar_try_wait(&ms.wfull[ws], (wit / kSmNW) & 1)) {
        sm_ev_mma(p, evi, SEV_WEIGHTS_READY, gi);
      } else {
        if (!mwait(p, &ms.wfull[ws], (wit / kSmNW) & 1)) goto out;
        sm_ev_mma(p, evi, SEV_WEIGHTS, gi);
      }
      if (nimg > 1 && !mwait(p, &ms.wfull[(wit + 1) % kSmNW], ((wit + 1) / kSmNW) & 1)) goto out;
      if (!mwait(p, &ms.ofull[os], ouse[os] & 1)) goto out;
      if (first && seg >= 2 && !mwait(p, &ms.accempty[tb], ((seg >> 1) - 1) & 1)) goto out;
      tc_fence_after();
      for (uint32_t img = 0; img < nimg; ++img) {
        const uint32_t a0 = smem_u32(smem + kSmOffW + ((wit + img) % kSmNW) * kSmWSlot);
        const uint32_t b0 = smem_u32(smem + kSmOffOp + os * obytes);
        const uint32_t d = ms.tmem_base + tb * 128;
#pragma unroll
        for (int j = 0; j < kKs / 16; ++j) {
          const uint64_t ad = smem_desc(a0 + uint32_t(j) * 2 * (kTileM / 8) * 128, (kTileM / 8) * 128, 128);
          const uint64_t bd = smem_desc(b0 + uint32_t(j) * 2 * blb, blb, 128);
          mma_f16(d, ad, bd, idesc, (first && img == 0 && j == 0) ? 0u : 1u);
        }
        mma_commit(&ms.wempty[(wit + img) % kSmNW]);
      }
      mma_commit(&ms.oempty[os]);
      if (last) {
        mma_commit(&ms.accfull[tb]);
        sm_ev_mma(p, evi, SEV_COMMIT, gi);
        ++seg;
      }
      wit += nimg;
      ++ouse[os];
    }
  }
out:
  // every MMA retires before TMEM and shared memory are released
  mma_commit(&ms.mmadone);
  mbar_wait(&ms.mmadone, 0);
}

// ------------------------------------------------------ consumer helpers
__device__ __forceinline__ void ld8f(const float* src, float (&v)[8]) {
  const float4 a = __ldcg(reinterpret_cast<const float4*>(src)), b = __ldcg(reinterpret_cast<const float4*>(src + 4));
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ uint4 pack8h(const float (&v)[8]) {
  const uint2 a = pack4_f16(v[0], v[1], v[2], v[3]), b = pack4_f16(v[4], v[5], v[6], v[7]);
  return make_uint4(a.x, a.y, b.x, b.y);
}

// The operand slices of units u0 .. u0+nu-1 (K slice u % n_ks: columns
// ks*128 .. +127) for the GEMM's R activation rows, each written to its ring
// slot as the K-major core-matrix image [16 k groups][N/8 row groups][8 rows]
// [8 k] of f16 (all consumer threads; one thread per 8 consecutive columns
// of a row, so global reads coalesce, and every unit's loads in one pass).
// i0: the run index of unit u0 (its operand goes to slot (i0 + ui) % slots).
template <int KIND>
__device__ void sm_build(const SParams& p, const SG& g, int gi, int u0, int nu, int i0, uint8_t* smem) {
  const int n8 = g.N / 8, per = g.R * 16;
  const uint32_t nop = sm_op_slots(g), obytes = sm_op_bytes(g);
  for (int it = threadIdx.x; it < nu * per; it += kSmConsumers) {
    const int ui = it / per, rem = it - ui * per;
    const int n = rem >> 4, k8 = rem & 15, k = ((u0 + ui) % g.n_ks) * kKs + k8 * 8;
    uint16_t* dst = reinterpret_cast<uint16_t*>(smem + kSmOffOp + (uint32_t(i0 + ui) % nop) * obytes);
    uint4 h;
    int rx = 0;   // the row's range exponent (H rows and residual rows), loaded alongside its values
    if (KIND == S_O) {
      h = __ldcg(reinterpret_cast<const uint4*>(p.a_o + size_t(n) * p.qw + k));
    } else {
      float v[8];
      if (KIND == S_PROJ) {
        // rows 2b, 2b+1: the Talker state H_b and the embedding of q0_b, the
        // first two positions of frame b (H and q0 feed the residual loop:
        // "拆解 Qwen3-TTS：OpenVINO 移植过程中的图分离与调度实践", section 1;
        // their order is a reading)
        const int b = n >> 1;
        if (g.k > 1) {
          // step k >= 2 with Talker-wide code tables: row n is E[k-2][the frame's input code]
          const int32_t c = p.in_code[size_t(g.k - 1) * p.B + n];
          const int kt = sm_mode(p) == SM_STEP ? p.row_step[n] : g.k;   // the row's own step in SM_STEP
          const uint4 e = *reinterpret_cast<const uint4*>(p.embed[kt - 2] + size_t(c) * p.th + k);
          const uint32_t w[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) { v[2 * i] = e16_to_f32(w[i], p.embed_f16); v[2 * i + 1] = e16_to_f32(w[i] >> 16, p.embed_f16); }
        } else if ((n & 1) == 0) {
          rx = __ldcg(sm_rexp(p, gi, n));
          const float4 a = __ldg(reinterpret_cast<const float4*>(p.H + size_t(b) * p.th + k));
          const float4 c = __ldg(reinterpret_cast<const float4*>(p.H + size_t(b) * p.th + k + 4));
          v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
        } else {
          int q = p.q0[b];
          q = q < 0 ? 0 : (q >= p.q0_vocab ? p.q0_vocab - 1 : q);   // reported by the step-1 input pass
          const uint4 e = __ldg(reinterpret_cast<const uint4*>(p.e0 + size_t(q) * p.th + k));
          const uint32_t w[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) { v[2 * i] = e16_to_f32(w[i], p.embed_f16); v[2 * i + 1] = e16_to_f32(w[i] >> 16, p.embed_f16); }
        }
      } else if (KIND == S_DOWN) {
        float u[8];
        ld8f(p.acc_gu + size_t(n) * 2 * p.F + k, v);
        ld8f(p.acc_gu + size_t(n) * 2 * p.F + p.F + k, u);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = silu_f(v[i]) * u[i];
      } else {
        // x * w_norm of an RMS-normalised input; the row scale is applied to
        // the GEMM's partial products instead
        const float* wn;
        int row = n, gr = n;   // the residual row; the GEMM's row
        if (kQkv<KIND>) wn = p.layer[g.l].attn_norm;
        else if (KIND == S_GU) wn = p.layer[g.l].ffn_norm;
        else {   // head: each frame's last position
          wn = p.out_norm;
          int r0 = 0, R = g.R;
          if (sm_grouped(p, g)) sm_rows(p, g, (u0 + ui) / g.n_ks, r0, R);
          if (n >= R) continue;   // rows past the tile's group: their outputs are not read
          row = g.k == 1 ? 2 * n + 1 : r0 + n;
          gr = r0 + n;
        }
        // the loads in flight together
        rx = __ldcg(sm_rexp(p, gi, gr));
        const float4 w0 = __ldg(reinterpret_cast<const float4*>(wn + k));
        const float4 w1 = __ldg(reinterpret_cast<const float4*>(wn + k + 4));
        ld8f(p.x + size_t(row) * p.d + k, v);
        const float w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] *= w[i];
      }
      if (kRange<KIND>) {
        const float sc = exp2i(-rx);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] *= sc;
      }
      h = pack8h(v);
    }
    *reinterpret_cast<uint4*>(dst + (size_t(k8 * n8 + (n >> 3)) << 6) + ((n & 7) << 3)) = h;
  }
}

// Per-warp sums of squares of rows r0 .. r0+ROWS-1 (those below R) of the
// GEMM's input into ms.ssp[warp]: each thread sums its columns of all ROWS
// rows with all of those loads in flight.  Up to 8 rows, one warp reduction
// per row present; 16 rows meet in one reduce-scatter across the warp.
template <int KIND, int ROWS>
__device__ __forceinline__ void sm_ssq(const SParams& p, const SG& g, SMisc& ms, int r0) {
  static_assert(ROWS == 8 || ROWS == 16, "8 rows reduce per row, 16 by reduce_scatter16");
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31, nc = p.d / 4;
  float sq[ROWS];
#pragma unroll
  for (int u = 0; u < ROWS; ++u) sq[u] = 0.f;
  for (int c = t; c < nc; c += kSmConsumers) {
    float4 a[ROWS];
#pragma unroll
    for (int u = 0; u < ROWS; ++u) {
      const int n = r0 + u, row = (KIND == S_HEAD && g.k == 1) ? 2 * n + 1 : n;
      a[u] = n < g.R ? __ldcg(reinterpret_cast<const float4*>(p.x + size_t(row) * p.d) + c)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < ROWS; ++u) sq[u] += a[u].x * a[u].x + a[u].y * a[u].y + a[u].z * a[u].z + a[u].w * a[u].w;
  }
  if constexpr (ROWS == 16) {
    // lanes 2i and 2i + 1 end with row r0 + i's warp total
    const float v = reduce_scatter16(sq, lane);
    if ((lane & 1) == 0 && r0 + (lane >> 1) < g.R) ms.ssp[warp][r0 + (lane >> 1)] = v;
  } else {
#pragma unroll
    for (int u = 0; u < ROWS; ++u) {
      if (r0 + u < g.R) {   // warp-uniform
        const float v = warp_sum(sq[u]);
        if (lane == 0) ms.ssp[warp][r0 + u] = v;
      }
    }
  }
}

// inv[n] = 1 / RMS of the GEMM's input row n, from the complete residual row
// (all consumer threads; the warps' partial sums meet in shared memory).  The
// caller's next barrier publishes ms.inv.
// The factor also undoes the operand's range scaling (times 2^e).  The
// gate/up GEMM's first CTA (record) writes the range exponent of each row
// for the GEMM after down, the next layer's QKV or the step's head, whose
// input row has grown from this one by the down projection only.
template <int KIND>
__device__ void sm_inv(const SParams& p, const SG& g, int gi, SMisc& ms, bool record) {
  const int t = threadIdx.x;
  if (g.R <= 8) {
    sm_ssq<KIND, 8>(p, g, ms, 0);
  } else {
    for (int r0 = 0; r0 < g.R; r0 += 16) sm_ssq<KIND, 16>(p, g, ms, r0);
  }
  named_bar(SBAR_CONS, kSmConsumers);
  if (t < g.R) {
    float ss = 0.f;
#pragma unroll
    for (int w = 0; w < kSmConsumerWarps; ++w) ss += ms.ssp[w][t];
    ms.inv[t] = rsqrtf(ss / float(p.d) + p.eps) * exp2i(__ldcg(sm_rexp(p, gi, t)));
    if (KIND == S_GU && record) {
      const int e = range_exp(ss / float(p.d));
      if (g.l + 1 < p.L || g.k > 1 || sm_mode(p) == SM_STEP) *sm_rexp(p, gi + 2, t) = e;
      else if (t & 1) *sm_rexp(p, gi + 2, t >> 1) = e;   // step 1's head reads rows 2b+1 as row b
    }
  }
}

// Add one segment's accumulator (tile mt, nsl K slices) into the GEMM's
// destination, scaled by the rows' inv for a normalised input.  Each warp
// drains 32 accumulator rows (output features) x 8 columns (activation rows)
// at a time, transposes them through its 1 KB of shared memory and adds 4
// consecutive features per thread with one vector reduction.
template <int KIND>
__device__ bool sm_drain(const SParams& p, SMisc& ms, uint8_t* smem, const SG& g, int gi, int mt, int nsl,
                         uint32_t& seg, bool publish, bool publish_first = false) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const uint32_t tb = seg & 1;
  if (t == 0) ms.flag[1] = mwait(p, &ms.accfull[tb], (seg >> 1) & 1);
  named_bar(SBAR_CONS, kSmConsumers);
  if (!ms.flag[1]) return false;
  if (t == 0) sm_ev(p, &ms.evc, SEV_ACC, gi);
  tc_fence_after();
  const int quarter = warp & 3, half = warp >> 2, cols = g.N / 2;
  int r0, R;
  sm_rows(p, g, mt, r0, R);
  // a grouped head's tile mt is tile mt % (V / 128) of its group's logits
  const int m0 = (sm_grouped(p, g) ? mt % (p.V / kTileM) : mt) * kTileM + quarter * 32;
  float* tp = reinterpret_cast<float*>(smem + kSmOffKeys) + warp * 256;   // [8 rows][32 features]
  for (int col = half * cols; col < (half + 1) * cols && col < R; col += 8) {   // warp-uniform bounds
    float v[8];
    tmem_ld8(ms.tmem_base + tb * 128 + (uint32_t(quarter * 32) << 16) + uint32_t(col), v);
#pragma unroll
    for (int i = 0; i < 8; ++i) tp[i * 32 + lane] = v[i];
    __syncwarp();
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
      const int f = pass * 4 + (lane >> 3), k4 = (lane & 7) * 4, n = col + f;
      if (n < R) {
        float4 x = *reinterpret_cast<const float4*>(tp + f * 32 + k4);
        if (sm_scaled<KIND>(g) || (KIND == S_PROJ && g.k == 1)) {
          const float s = ms.inv[r0 + n];
          x.x *= s; x.y *= s; x.z *= s; x.w *= s;
        }
        red_add_v4_f32(g.out + size_t(r0 + n) * g.ld + m0 + k4, x);
      }
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(&ms.accempty[tb]);
  ++seg;
  if (publish) {
    named_bar(SBAR_CONS, kSmConsumers);
    if (t == 0) {
      // release: the bar.sync above orders every consumer thread's reductions first
      fence_acq_rel_gpu();   // one fence releases the reductions for both counts
      if (gi != p.withhold || !publish_first) {   // a test of the failure path makes one count go missing
        if (kQkv<KIND>) red_relaxed_add(sm_qkv_tile(p, g.k, g.l, mt), unsigned(nsl));
        red_relaxed_add(sm_done(p, gi), unsigned(nsl));
      }
      sm_ev(p, &ms.evc, SEV_PUBLISHED, gi);
    }
  }
  return true;
}

// This CTA's units of GEMM gi (all consumer threads): wait for the operand's
// source, build the operand slices, drain the accumulators.
//
// When the whole run fits in the operand ring (the usual case) every unit is
// built in one pass, so the MMAs of all segments start together, and the
// drained segments are released with one counter update.  Otherwise each
// segment is built and then the previous one drained, so that a segment's
// MMAs wait only for drains two segments back, which precede the builds they
// follow, and the ring's waits are for MMAs of units built earlier: neither
// can wait on work that comes later in this order.
template <int KIND>
__device__ bool sm_gemm(const SParams& p, SMisc& ms, uint8_t* smem, int gi, uint32_t& seg) {
  const SG g = sgemm(p, gi);
  int beg, end;
  sm_run(g, gi, beg, end);
  if (beg >= end) return true;
  const int t = threadIdx.x;
  if (t == 0) {
    const unsigned* ctr;
    unsigned want;
    sm_ready(p, gi, ctr, want);
    ms.flag[2] = poll_geq(p, ctr, want);
  }
  named_bar(SBAR_CONS, kSmConsumers);
  if (!ms.flag[2]) return false;
  if (t == 0) sm_ev(p, &ms.evc, SEV_READY, gi);
  const uint32_t nop = sm_op_slots(g);
  // builds units [u, u_end) in passes of at most one ring
  auto build = [&](int u, int u_end) -> bool {
    while (u < u_end) {
      const int nu = min(u_end - u, int(nop));
      if (t == 0) {
        // A slot is free once the MMAs of the unit that used it last have
        // completed.  For a unit of an earlier GEMM that is already known:
        // this CTA drained its accumulator, which the MMAs' commit gates.
        // Within this run, wait for the unit one ring earlier.
        bool ok = true;
        for (int i = 0; i < nu && ok; ++i) {
          const uint32_t ri = uint32_t(u + i - beg), os = ri % nop;
          if (ri >= nop) ok = mwait(p, &ms.oempty[os], (ms.ouse[os] - 1) & 1);
        }
        ms.flag[3] = ok;
      }
      named_bar(SBAR_CONS, kSmConsumers);
      if (!ms.flag[3]) return false;
      sm_build<KIND>(p, g, gi, u, nu, u - beg, smem);
      fence_proxy_async_shared();   // the tensor cores read what these generic stores wrote
      named_bar(SBAR_CONS, kSmConsumers);
      if (t == 0)
        for (int i = 0; i < nu; ++i) {
          const uint32_t os = uint32_t(u + i - beg) % nop;
          mbar_arrive(&ms.ofull[os]);
          ++ms.ouse[os];
        }
      u += nu;
    }
    if (t == 0) sm_ev(p, &ms.evc, SEV_BUILT, gi);
    return true;
  };
  auto scale = [&]() {
    if (sm_scaled<KIND>(g)) {
      sm_inv<KIND>(p, g, gi, ms, beg == 0);
      named_bar(SBAR_CONS, kSmConsumers);
    } else if (KIND == S_PROJ && g.k == 1) {
      // unscaled, but the H rows carry range exponents
      for (int n = t; n < g.R; n += kSmConsumers) ms.inv[n] = exp2i(__ldcg(sm_rexp(p, gi, n)));
      named_bar(SBAR_CONS, kSmConsumers);
    }
  };
  if (end - beg <= int(nop)) {
    if (!build(beg, end)) return false;
    scale();
    for (int s = beg; s < end;) {
      const int ks0 = s % g.n_ks, seg_end = min(end, s + (g.n_ks - ks0));
      if (!sm_drain<KIND>(p, ms, smem, g, gi, s / g.n_ks, seg_end - s, seg, false)) return false;
      s = seg_end;
    }
    named_bar(SBAR_CONS, kSmConsumers);
    if (t == 0) {
      // release: the bar.sync above orders every consumer thread's reductions
      // first, and one fence releases them for every count below
      fence_acq_rel_gpu();
      if (gi == p.withhold && beg == 0) return true;   // a test of the failure path makes the counts go missing
      if (kQkv<KIND>)
        for (int s = beg; s < end;) {
          const int ks0 = s % g.n_ks, seg_end = min(end, s + (g.n_ks - ks0));
          red_relaxed_add(sm_qkv_tile(p, g.k, g.l, s / g.n_ks), unsigned(seg_end - s));
          s = seg_end;
        }
      red_relaxed_add(sm_done(p, gi), unsigned(end - beg));
      sm_ev(p, &ms.evc, SEV_PUBLISHED, gi);
    }
    return true;
  }
  int s = beg, si = 0, prev_mt = -1, prev_nsl = 0;
  while (s < end) {
    const int ks0 = s % g.n_ks, mt = s / g.n_ks;
    const int seg_end = min(end, s + (g.n_ks - ks0)), nsl = seg_end - s;
    if (!build(s, seg_end)) return false;
    if (si == 0) scale();
    if (si > 0 && !sm_drain<KIND>(p, ms, smem, g, gi, prev_mt, prev_nsl, seg, true, si == 1 && beg == 0)) return false;
    prev_mt = mt;
    prev_nsl = nsl;
    ++si;
    s = seg_end;
  }
  return sm_drain<KIND>(p, ms, smem, g, gi, prev_mt, prev_nsl, seg, true, si == 1 && beg == 0);
}

// Step-1 setup, one warp per row r < 2B: the residual row starts at the
// projection bias (the projection's partials are added to it); the row of
// both q|k|v accumulators and the frame's logit row start at zero;
// out-of-range first codes are reported.  An H row's range exponent, from
// its mean square, serves the projection's operand row and, as the
// reference of the projection's output, layer 0's QKV operand row.
__device__ bool sm_prep1(const SParams& p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, G = gridDim.x;
  const int qkvw = p.qw + 2 * p.kvw;
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int r = blockIdx.x + warp * G; r < 2 * p.B; r += kSmConsumerWarps * G) {
    for (int f = lane * 4; f < p.d; f += 128)
      *reinterpret_cast<float4*>(p.x + size_t(r) * p.d + f) = *reinterpret_cast<const float4*>(p.b_proj + f);
    for (int f = lane * 4; f < qkvw; f += 128) {
      *reinterpret_cast<float4*>(p.acc_qkv[0] + size_t(r) * qkvw + f) = z4;
      *reinterpret_cast<float4*>(p.acc_qkv[1] + size_t(r) * qkvw + f) = z4;
    }
    if (r < p.B)
      for (int f = lane * 4; f < p.V; f += 128) *reinterpret_cast<float4*>(p.logits + size_t(r) * p.V + f) = z4;
    if ((r & 1) && lane == 0) {
      const int q = p.q0[r >> 1];
      if (q < 0 || q >= p.q0_vocab) set_status(p.status, QP_ERR_BAD_TOKEN);
    }
    if ((r & 1) == 0) {
      const float* hr = p.H + size_t(r >> 1) * p.th;
      float ss = 0.f;
      for (int f = lane * 4; f < p.th; f += 128) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(hr + f));
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
      }
      const int e = range_exp(warp_sum(ss) / float(p.th));
      if (lane == 0) {
        *sm_rexp(p, 0, r) = e;
        *sm_rexp(p, sgi_of(p, 1, 0, 0), r) = e;
      }
    }
    __syncwarp();
    if (lane == 0) red_release_add(sm_prep(p, 1), 1u);
  }
  return true;
}

// 1/RMS of residual row `row` (all consumer threads; the same value in
// every thread).  ms.ssp[*][0] holds the warps' partial sums until the
// caller's next consumer barrier.
__device__ float sm_row_inv(const SParams& p, SMisc& ms, int row) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  float ss = 0.f;
  for (int c = t * 4; c < p.d; c += 4 * kSmConsumers) {
    const float4 v = __ldcg(reinterpret_cast<const float4*>(p.x + size_t(row) * p.d + c));
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = warp_sum(ss);
  if (lane == 0) ms.ssp[warp][0] = ss;
  named_bar(SBAR_CONS, kSmConsumers);
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kSmConsumerWarps; ++w) tot += ms.ssp[w][0];
  return rsqrtf(tot / float(p.d) + p.eps);
}

// The code of step `step` for frame b, computed by the whole CTA (all
// consumer threads; the same value, or -1 if the grid aborted, in every
// thread).  Greedy: the argmax of the frame's complete logit row (lowest
// index on ties; from step 2 on the row holds the logits before the row
// scale), which is copied out, scaled, if asked and zeroed for the next
// step's accumulation.
// Sampling: the decision the sampling pass published.
__device__ int sm_code(const SParams& p, SMisc& ms, int step, int b) {
  // the head GEMM that produced row b's logits, and where the call's outputs go
  const int gih = sgi_head(p, step);
  int out_row = b, out_step = step - sm_k_first(p);
  if (sm_mode(p) == SM_STEP) {   // one step per row, in the caller's row order
    out_row = p.row_perm[b];
    out_step = 0;
  }
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  if (sm_sampled(p)) {
    if (t == 0) {
      unsigned* dp = p.decided + size_t(step - 1) * p.B + b;
      ms.bcast = poll_geq(p, dp, 1u) ? int(ld_acquire_u32(dp)) - 1 : -1;
    }
    named_bar(SBAR_CONS, kSmConsumers);
    const int code = ms.bcast;
    named_bar(SBAR_CONS, kSmConsumers);
    return code;
  }
  if (t == 0) {
    const SG h = sgemm(p, gih);
    ms.bcast = poll_geq(p, sm_done(p, gih), unsigned(h.n_mt * h.n_ks)) ? 0 : -1;
  }
  named_bar(SBAR_CONS, kSmConsumers);
  if (ms.bcast < 0) return -1;
  float* row = p.logits + size_t(b) * p.V;
  float* dst = p.out_logits ? p.out_logits + (size_t(out_row) * sm_n_run(p) + out_step) * p.V : nullptr;
  // the head's input row scale, and the range factor of its operand row
  const float rs = dst && step > 1 ? sm_row_inv(p, ms, b) * exp2i(__ldcg(sm_rexp(p, gih, b))) : 1.f;
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  unsigned long long best = 0ull;
  for (int f0 = t * 4; f0 < p.V; f0 += 2 * 4 * kSmConsumers) {
    float4 v[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int f = f0 + i * 4 * kSmConsumers;
      v[i] = f < p.V ? __ldcg(reinterpret_cast<const float4*>(row + f)) : z4;
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int f = f0 + i * 4 * kSmConsumers;
      if (f >= p.V) continue;
      if (dst) *reinterpret_cast<float4*>(dst + f) = make_float4(v[i].x * rs, v[i].y * rs, v[i].z * rs, v[i].w * rs);
      *reinterpret_cast<float4*>(row + f) = z4;
      unsigned long long c = pack_argmax(v[i].x, f);
      const unsigned long long c1 = pack_argmax(v[i].y, f + 1), c2 = pack_argmax(v[i].z, f + 2),
                               c3 = pack_argmax(v[i].w, f + 3);
      c = c1 > c ? c1 : c;
      c = c2 > c ? c2 : c;
      c = c3 > c ? c3 : c;
      best = c > best ? c : best;
    }
  }
  best = warp_max_u64(best);
  if (lane == 0) ms.redu[warp] = best;
  named_bar(SBAR_CONS, kSmConsumers);
  unsigned long long v = ms.redu[0];
#pragma unroll
  for (int i = 1; i < kSmConsumerWarps; ++i) v = ms.redu[i] > v ? ms.redu[i] : v;
  named_bar(SBAR_CONS, kSmConsumers);   // ms.redu and ms.bcast are reused
  return unpack_argmax_index(v);
}

// SM_STEP inputs, one row per CTA: row b (the caller's row row_perm[b]) is
// at step row_step[b], and its input code comes from the caller.  The
// residual row starts at the row's code embedding (or, with Talker-wide
// tables, at the projection's bias, the code recorded for the projection);
// the row of both q|k|v accumulators and the logit row start at zero.
__device__ bool sm_prep_step(const SParams& p, SMisc& ms) {
  const int t = threadIdx.x, G = gridDim.x, qkvw = p.qw + 2 * p.kvw;
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int b = (blockIdx.x + 3) % G; b < p.B; b += G) {
    if (t == 0) {
      int c = p.code_in[p.row_perm[b]];
      if (c < 0 || c >= p.V) {
        set_status(p.status, QP_ERR_BAD_TOKEN);
        c = c < 0 ? 0 : p.V - 1;
      }
      ms.bcast = c;
      if (p.proj_in) p.in_code[size_t(1) * p.B + b] = c;   // read by the step's projection (k = 2 slot)
    }
    named_bar(SBAR_CONS, kSmConsumers);
    const int c = ms.bcast;
    const uint16_t* e = p.embed[p.row_step[b] - 2] + size_t(c) * p.d;
    for (int f = t * 4; f < p.d; f += 4 * kSmConsumers) {
      float4 v;
      if (p.proj_in) {
        v = *reinterpret_cast<const float4*>(p.b_proj + f);
      } else {
        const uint2 ev = *reinterpret_cast<const uint2*>(e + f);
        v = make_float4(e16_to_f32(ev.x, p.embed_f16), e16_to_f32(ev.x >> 16, p.embed_f16),
                        e16_to_f32(ev.y, p.embed_f16), e16_to_f32(ev.y >> 16, p.embed_f16));
      }
      *reinterpret_cast<float4*>(p.x + size_t(b) * p.d + f) = v;
    }
    for (int f = t * 4; f < qkvw; f += 4 * kSmConsumers) {
      *reinterpret_cast<float4*>(p.acc_qkv[0] + size_t(b) * qkvw + f) = z4;
      *reinterpret_cast<float4*>(p.acc_qkv[1] + size_t(b) * qkvw + f) = z4;
    }
    for (int f = t * 4; f < p.V; f += 4 * kSmConsumers) *reinterpret_cast<float4*>(p.logits + size_t(b) * p.V + f) = z4;
    named_bar(SBAR_CONS, kSmConsumers);   // the release below follows every thread's stores; ms.bcast is reused
    if (t == 0) red_release_add(sm_prep(p, 2), 1u);
  }
  return true;
}

// Step k >= 2 inputs, one frame per CTA: report the previous step's code,
// embed the next input (teacher-forced if asked) as residual row b.  With
// Talker-wide code tables the row starts at the projection's bias instead
// and the code is recorded for the projection's operand build.
__device__ bool sm_prepk(const SParams& p, SMisc& ms, int k) {
  if (kSmSlots) return sm_prep_step(p, ms);   // that kernel reaches step k >= 2 in SM_STEP calls only
  const int t = threadIdx.x, G = gridDim.x;
  for (int b = (blockIdx.x + k * 11) % G; b < p.B; b += G) {
    const int code = sm_code(p, ms, k - 1, b);
    if (code < 0) return false;
    if (t == 0) {
      p.out_codes[size_t(b) * sm_n_run(p) + (k - 1 - sm_k_first(p))] = code;
      int nc = p.forced ? p.forced[size_t(b) * p.n_steps + (k - 2)] : code;
      if (nc < 0 || nc >= p.V) {
        set_status(p.status, QP_ERR_BAD_TOKEN);
        nc = nc < 0 ? 0 : p.V - 1;
      }
      ms.bcast = nc;
    }
    named_bar(SBAR_CONS, kSmConsumers);
    if (p.proj_in) {
      if (t == 0) p.in_code[size_t(k - 1) * p.B + b] = ms.bcast;
      for (int f = t * 4; f < p.d; f += 4 * kSmConsumers)
        *reinterpret_cast<float4*>(p.x + size_t(b) * p.d + f) = *reinterpret_cast<const float4*>(p.b_proj + f);
      named_bar(SBAR_CONS, kSmConsumers);
      if (t == 0) red_release_add(sm_prep(p, k), 1u);
      continue;
    }
    const uint16_t* e = p.embed[k - 2] + size_t(ms.bcast) * p.d;
    for (int f = t * 4; f < p.d; f += 4 * kSmConsumers) {
      const uint2 ev = *reinterpret_cast<const uint2*>(e + f);
      *reinterpret_cast<float4*>(p.x + size_t(b) * p.d + f) =
          make_float4(e16_to_f32(ev.x, p.embed_f16), e16_to_f32(ev.x >> 16, p.embed_f16), e16_to_f32(ev.y, p.embed_f16),
                      e16_to_f32(ev.y >> 16, p.embed_f16));
    }
    named_bar(SBAR_CONS, kSmConsumers);
    if (t == 0) red_release_add(sm_prep(p, k), 1u);
  }
  return true;
}

// The codes of the call's last step (in SM_STEP each row's own step).
__device__ bool sm_final(const SParams& p, SMisc& ms) {
  const int G = gridDim.x, k_last = sm_k_first(p) + sm_n_run(p) - 1;
  for (int b = (blockIdx.x + 5) % G; b < p.B; b += G) {
    const int code = sm_code(p, ms, sm_mode(p) == SM_STEP ? p.row_step[b] : k_last, b);
    if (code < 0) return false;
    const int out_row = sm_mode(p) == SM_STEP ? p.row_perm[b] : b;
    if (threadIdx.x == 0) p.out_codes[size_t(out_row) * sm_n_run(p) + (sm_n_run(p) - 1)] = code;
  }
  return true;
}

// Attention of one (frame, kv head) per warp at layer l of step k: the row
// scale 1/RMS of the layer's input row (the QKV projection's partials are
// added unscaled; the residual row is unchanged until the O projection,
// which waits for every item), per-head RMSNorm and RoPE of the new
// position(s), KV append, causal softmax over positions 0..pos for the
// group's q heads, output into the O operand rows.
// Lane l holds dims 4l..4l+3 of every 128-vector; the scores of two q heads x
// 16 positions are 32 partial dot products per lane, summed across the warp
// by one reduce-scatter that leaves score (head l/16, position l%16) in lane
// l.  The item then zeroes what it read of the q|k|v accumulator and its
// share of the frame's gate|up accumulator rows, which this layer's GEMMs
// accumulate into next.
__device__ bool sm_attn(const SParams& p, SMisc& ms, int k, int l) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, G = gridDim.x;
  const int P = k == 1 ? 2 : 1, pos0 = k == 1 ? 0 : k;
  const int gi_q = sgi_of(p, k, l, 0);
  const int qkvw = p.qw + 2 * p.kvw, grp = p.n_q / p.n_kv, ctx = p.n_steps + 1;
  const SLayer& L = p.layer[l];
  const int n_items = p.B * p.n_kv;
  const unsigned slices = unsigned(p.d / kKs);
  const int guw = ((2 * p.F + p.n_kv - 1) / p.n_kv + 3) & ~3;   // gate|up columns zeroed per item
  const float scale = rsqrtf(float(kHeadDim));
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  uint16_t* kvl = p.kv + size_t(l) * p.Bmax * ctx * 2 * p.kvw;
  for (int i = (blockIdx.x + gi_q * 13) % G + warp * G; i < n_items; i += kSmConsumerWarps * G) {
    const int b = i / p.n_kv, j = i % p.n_kv, r0 = b * P;
    // the group's q head tiles, its k tile and its v tile: one lane polls each
    int okl = 1;
    if (lane < grp + 2) {
      const int tile = lane < grp ? j * grp + lane : (lane == grp ? p.qw / kHeadDim + j : (p.qw + p.kvw) / kHeadDim + j);
      okl = poll_geq(p, sm_qkv_tile(p, k, l, tile), slices);
    }
    if (!__all_sync(0xffffffffu, okl)) return false;
    __syncwarp();   // every lane's reads follow the acquires
    if (lane == 0) sm_ev(p, &ms.evc, SEV_ATT_READY, gi_q);
    // the frame's KV state (its slot in state-slot calls) and first new position (its own step in SM_STEP)
    uint16_t* kvb = kvl + size_t(sm_slot(p, b)) * ctx * 2 * p.kvw + j * kHeadDim + lane * 4;   // + (pos*2 + {0,1}) * kvw
    const int pos_b = sm_mode(p) == SM_STEP ? p.row_step[b] : pos0;
    for (int pp = 0; pp < P; ++pp) {
      const int r = r0 + pp, pos = pos_b + pp;
      float* row = p.acc_qkv[((k - 1) * p.L + l) & 1] + size_t(r) * qkvw;
      float* kr = row + p.qw + j * kHeadDim + lane * 4;
      float* vr = row + p.qw + p.kvw + j * kHeadDim + lane * 4;
      // independent loads first: the input row, new k, v, the first two q heads, then the cache
      // the QKV operand row's range exponent (its partials were added unscaled)
      const int rx = __ldcg(sm_rexp(p, gi_q, r));
      float ss = 0.f;
#pragma unroll 8
      for (int c = lane * 4; c < p.d; c += 128) {
        const float4 xv = __ldcg(reinterpret_cast<const float4*>(p.x + size_t(r) * p.d + c));
        ss += xv.x * xv.x + xv.y * xv.y + xv.z * xv.z + xv.w * xv.w;
      }
      float4 kraw = __ldcg(reinterpret_cast<const float4*>(kr));
      float4 vnew = __ldcg(reinterpret_cast<const float4*>(vr));
      float4 qraw[2];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
        qraw[hh] = hh < grp ? __ldcg(reinterpret_cast<const float4*>(row + (j * grp + hh) * kHeadDim + lane * 4)) : z4;
      const float ms_x = warp_sum(ss) / float(p.d);
      const float rs = rsqrtf(ms_x + p.eps) * exp2i(rx);
      // this row's range exponent for the gate/up operand, whose input row
      // grows from this one by the O projection only
      if (j == 0 && lane == 0) *sm_rexp(p, sgi_of(p, k, l, 2), r) = range_exp(ms_x);
      kraw.x *= rs; kraw.y *= rs; kraw.z *= rs; kraw.w *= rs;
      vnew.x *= rs; vnew.y *= rs; vnew.z *= rs; vnew.w *= rs;
      uint2 kh[kMaxCtx], vh[kMaxCtx];
#pragma unroll
      for (int t = 0; t < kMaxCtx; ++t) {
        kh[t] = t < pos ? __ldcg(reinterpret_cast<const uint2*>(kvb + (size_t(t) * 2 + 0) * p.kvw)) : make_uint2(0, 0);
        if (!kSmSlots)
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
            float* qr = row + (j * grp + g0 + hh) * kHeadDim + lane * 4;
            float4 q = g0 == 0 ? qraw[hh] : __ldcg(reinterpret_cast<const float4*>(qr));
            q.x *= rs; q.y *= rs; q.z *= rs; q.w *= rs;
            qn[hh] = norm_rope(q, L.q_norm, p.eps, p.rope_cs + pos * 64, lane);
            *reinterpret_cast<float4*>(qr) = z4;
          }
        }
        float part[32];
#pragma unroll
        for (int t = 0; t < kMaxCtx; ++t) {
          part[t] = part[16 + t] = 0.f;
          if (t <= pos) {   // later positions are masked; pos is the same in every lane
            const float4 kk = t < pos ? unpack4_f16(kh[t]) : knew;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
              part[hh * 16 + t] = qn[hh].x * kk.x + qn[hh].y * kk.y + qn[hh].z * kk.z + qn[hh].w * kk.w;
          }
        }
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
        // the state-slot kernel loads the values here, after the scores: its
        // rows' positions differ, and holding both caches across the softmax
        // spills registers there
        if (kSmSlots)
#pragma unroll
          for (int t = 0; t < kMaxCtx; ++t)
            vh[t] = t < pos ? __ldcg(reinterpret_cast<const uint2*>(kvb + (size_t(t) * 2 + 1) * p.kvw)) : make_uint2(0, 0);
#pragma unroll
        for (int t = 0; t < kMaxCtx; ++t) {
          if (t <= pos) {
            const float4 vv = t < pos ? unpack4_f16(vh[t]) : vnew;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const float w = __shfl_sync(0xffffffffu, pr, hh * 16 + t);
              o2[hh].x += w * vv.x; o2[hh].y += w * vv.y; o2[hh].z += w * vv.z; o2[hh].w += w * vv.w;
            }
          }
        }
        for (int hh = 0; hh < nh; ++hh)
          *reinterpret_cast<uint2*>(p.a_o + size_t(r) * p.qw + (j * grp + g0 + hh) * kHeadDim + lane * 4) =
              pack4_f16(o2[hh].x, o2[hh].y, o2[hh].z, o2[hh].w);
      }
      for (int f = j * guw + lane * 4; f < min(2 * p.F, (j + 1) * guw); f += 128)
        *reinterpret_cast<float4*>(p.acc_gu + size_t(r) * 2 * p.F + f) = z4;
      __syncwarp();   // the next position of this frame reads what was stored here
    }
    __syncwarp();
    if (lane == 0) {
      red_release_add(sm_att(p, k, l), 1u);
      sm_ev(p, &ms.evc, SEV_ATT_DONE, gi_q);
    }
  }
  return true;
}

// Gumbel top-k decisions of step k: each half of the consumer warps (4
// warps) decides one frame, so a CTA takes two frames at a time (one, by
// half 0, when the vocabulary is too large for two key arrays).  The row's
// logits are the accumulated ones, times the head input row's scale (and
// its operand's range factor) from step 2 on.  The logit row is copied out
// if asked and zeroed for the next step.
__device__ bool sm_decide(const SParams& p, SMisc& ms, uint32_t* keys, int k) {
  constexpr int NG = kSmConsumers / 2;
  const int V = p.V, t = threadIdx.x, G = gridDim.x, half = t / NG, tg = t - half * NG;
  const int lane = tg & 31, w = tg >> 5;
  const bool two = 2 * V <= kMaxVocab;
  const int bar = SBAR_HALF0 + half, gih = sgi_head(p, k);
  const SG h = sgemm(p, gih);
  TopkScratch& sc = ms.topk[half];
  for (int b0 = (blockIdx.x + k * 7) % G; b0 < p.B; b0 += two ? 2 * G : G) {
    const int b = b0 + (two ? half * G : 0);
    if (b >= p.B || (!two && half == 1)) continue;   // warp-uniform: the half sits this frame out
    // In state-slot calls a row decides one step (its own, in SM_STEP), its
    // noise and logits are the caller's row row_perm[b], and the decision is
    // filed under the row's step.
    const bool slots = sm_mode(p) != SM_RUN;
    const int kd = sm_mode(p) == SM_STEP ? p.row_step[b] : k;
    const size_t orow = slots ? size_t(p.row_perm[b]) : size_t(b) * p.n_steps + (k - 1);
    if (tg == 0) ms.hflag[half] = poll_geq(p, sm_done(p, gih), unsigned(h.n_mt * h.n_ks));
    named_bar(bar, NG);
    if (!ms.hflag[half]) return false;
    float* l = p.logits + size_t(b) * V;
    float rs = 1.f;
    if (k > 1) {   // 1/RMS of the head's input row, by this half
      float ss = 0.f;
      for (int c = tg * 4; c < p.d; c += 4 * NG) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(p.x + size_t(b) * p.d + c));
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
      }
      ss = warp_sum(ss);
      if (lane == 0) sc.rsum[w] = ss;
      named_bar(bar, NG);
      float tot = 0.f;
#pragma unroll
      for (int i = 0; i < NG / 32; ++i) tot += sc.rsum[i];
      rs = rsqrtf(tot / float(p.d) + p.eps) * exp2i(__ldcg(sm_rexp(p, gih, b)));
    }
    const float* gb = p.gumbel + orow * V;
    const int code = gumbel_topk_group<NG>(l, rs, p.temperature, gb, V, p.top_k, keys + (two ? half * V : 0), sc,
                                           bar, tg);
    float* dst = p.out_logits ? p.out_logits + orow * V : nullptr;
    for (int i = tg; i < V; i += NG) {
      if (dst) dst[i] = __ldcg(l + i) * rs;
      l[i] = 0.f;
    }
    named_bar(bar, NG);
    if (tg == 0) {
      __threadfence();
      atomicExch(p.decided + size_t(kd - 1) * p.B + b, unsigned(code + 1));
    }
  }
  return true;
}

__device__ void sm_consumer(const SParams& p, SMisc& ms, uint8_t* smem) {
  uint32_t seg = 0;
  int sec = 0;
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + kSmOffKeys);
  // A section ends with one consumer-wide barrier; a failed wait in any warp
  // makes every consumer warp leave there together.
#define SM_SECTION(expr)                      \
  {                                           \
    sm_trace_mark(p, sec, 0);                 \
    const bool ok_ = (expr);                  \
    if (!ok_) ms.fail = 1;                    \
    named_bar(SBAR_CONS, kSmConsumers);       \
    sm_trace_mark(p, sec, 1);                 \
    ++sec;                                    \
    if (ms.fail) return;                      \
  }
  if (sm_mode(p) != SM_STEP) SM_SECTION(sm_prep1(p));
  for (int k = sm_k_first(p); k < sm_k_first(p) + sm_n_run(p); ++k) {
    if (k > 1) SM_SECTION(sm_prepk(p, ms, k));
    // one call site: a GEMM section inlined twice costs instruction fetch
    if (k == 1 || p.proj_in) SM_SECTION(sm_gemm<S_PROJ>(p, ms, smem, sgi_proj(p, k), seg));
    for (int l = 0; l < p.L; ++l) {
      SM_SECTION(sm_gemm<S_QKVU>(p, ms, smem, sgi_of(p, k, l, 0), seg));
      SM_SECTION(sm_attn(p, ms, k, l));
      SM_SECTION(sm_gemm<S_O>(p, ms, smem, sgi_of(p, k, l, 1), seg));
      SM_SECTION(sm_gemm<S_GU>(p, ms, smem, sgi_of(p, k, l, 2), seg));
      SM_SECTION(sm_gemm<S_DOWN>(p, ms, smem, sgi_of(p, k, l, 3), seg));
    }
    SM_SECTION(sm_gemm<S_HEAD>(p, ms, smem, sgi_head(p, k), seg));
    if (sm_sampled(p)) SM_SECTION(sm_decide(p, ms, keys, k));
  }
  SM_SECTION(sm_final(p, ms));
#undef SM_SECTION
}

// The greedy frame-loop kernel is k_frames_small, the sampling one
// k_frames_small_sampled, the state-slot kernel k_slots_small.
#if QP_SMALL_SLOTS && QP_SMALL_SAMPLED
#define SM_KERNEL k_slots_small_sampled
#elif QP_SMALL_SLOTS
#define SM_KERNEL k_slots_small
#elif QP_SMALL_SAMPLED
#define SM_KERNEL k_frames_small_sampled
#else
#define SM_KERNEL k_frames_small
#endif
__global__ void __launch_bounds__(kSmThreads, 1) SM_KERNEL(const SParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  SMisc& ms = *reinterpret_cast<SMisc*>(smem + kSmOffMisc);
  const int t = threadIdx.x, warp = t >> 5;
  if (t == 0) {
    for (int i = 0; i < kSmNW; ++i) { mbar_init(&ms.wfull[i], 1); mbar_init(&ms.wempty[i], 1); }
    for (int i = 0; i < kSmMaxOp; ++i) { mbar_init(&ms.ofull[i], 1); mbar_init(&ms.oempty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&ms.accfull[i], 1); mbar_init(&ms.accempty[i], kSmConsumerWarps); }
    mbar_init(&ms.mmadone, 1);
    ms.fail = 0;
    ms.evc = 0;
    for (int i = 0; i < kSmMaxOp; ++i) { ms.ouse[i] = 0; ms.ouse_m[i] = 0; }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(&ms.tmem_base, kSmTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp < kSmConsumerWarps) {
    sm_consumer(p, ms, smem);
  } else if (warp == kSmProducerWarp) {
    if ((t & 31) == 0) sm_producer(p, ms, smem);
    __syncwarp();
  } else if (warp == kSmMmaWarp) {
    if ((t & 31) == 0) sm_mma(p, ms, smem);
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(ms.tmem_base, kSmTmemCols);
}

// ----------------------------------------------------------------- host
size_t sm_al256(size_t b) { return (b + 255) & ~size_t(255); }

struct SmSync {
  size_t done, qkv_tile, att, prep, decided, in_code, rexp, abort_flag, total;
  int NGEMM, NHT;
};

// The sync region of a call.  The program: SM_RUN the whole frame loop;
// SM_BEGIN step 1 only; SM_STEP [the projection], 4 GEMMs per layer and the
// grouped head.
SmSync sm_sync_layout(const qp_geometry& g, int B, int mode = SM_RUN) {
  SmSync S{};
  const int proj_in = g.code_embed_dim != g.hidden;   // a projection GEMM per step k >= 2
  S.NGEMM = 1 + g.n_steps * (4 * g.layers + 1) + proj_in * (g.n_steps - 1);
  if (mode == SM_BEGIN) S.NGEMM = 1 + 4 * g.layers + 1;
  if (mode == SM_STEP) S.NGEMM = proj_in + 4 * g.layers + 1;
  S.NHT = g.n_q_heads + 2 * g.n_kv_heads;   // 128-row tiles of q|k|v (head_dim 128)
  const size_t steps = size_t(g.n_steps);
  size_t o = 0;
  S.done = o;       o += sm_al256(size_t(S.NGEMM) * 4);
  S.qkv_tile = o;   o += sm_al256(steps * g.layers * S.NHT * 4);
  S.att = o;        o += sm_al256(steps * g.layers * 4);
  S.prep = o;       o += sm_al256(steps * 4);
  S.decided = o;    o += sm_al256(steps * B * 4);
  S.in_code = o;    o += sm_al256(steps * B * 4);
  S.rexp = o;       o += sm_al256(size_t(S.NGEMM) * 2 * B * 4);
  S.abort_flag = o; o += 256;
  S.total = o;
  return S;
}

void sm_fill(SParams& p, const qp_handle* h, const RunArgs& a, uint8_t* scratch, const Scratch& L, uint8_t* sync,
             const SmSync& S, int bmax) {
  const qp_geometry& g = h->g;
  p.d = g.hidden; p.qw = g.n_q_heads * kHeadDim; p.kvw = g.n_kv_heads * kHeadDim; p.F = g.ffn; p.V = g.vocab;
  p.th = g.talker_hidden; p.L = g.layers; p.n_q = g.n_q_heads; p.n_kv = g.n_kv_heads; p.n_steps = g.n_steps;
  p.q0_vocab = g.q0_vocab; p.eps = g.rms_eps;
  // 16-bit matrices as packed; Q8_0 matrices through their f16 hi and lo images
  auto hi = [](const PackedMat& m) {
    return reinterpret_cast<const uint16_t*>(m.fmt == WF_Q8_0 ? m.w16[0] : m.w);
  };
  auto lo = [](const PackedMat& m) {
    return m.fmt == WF_Q8_0 ? reinterpret_cast<const uint16_t*>(m.w16[1]) : nullptr;
  };
  p.w_proj = hi(h->proj); p.w_proj_lo = lo(h->proj); p.b_proj = h->b_proj; p.e0 = h->e0;
  p.embed_f16 = h->embed_f16;
  for (int l = 0; l < g.layers; ++l) {
    const LayerW& Lw = h->layer[l];
    const PackedMat* mats[4] = {&Lw.qkv, &Lw.o, &Lw.gu, &Lw.down};
    for (int i = 0; i < 4; ++i) { p.layer[l].w[i] = hi(*mats[i]); p.layer[l].wl[i] = lo(*mats[i]); }
    p.layer[l].attn_norm = Lw.attn_norm; p.layer[l].q_norm = Lw.q_norm;
    p.layer[l].k_norm = Lw.k_norm; p.layer[l].ffn_norm = Lw.ffn_norm;
  }
  p.out_norm = h->out_norm;
  for (int j = 0; j < g.n_steps; ++j) {
    p.embed[j] = h->embed[j];
    p.w_head[j] = hi(h->head[j]);
    p.w_head_lo[j] = lo(h->head[j]);
  }
  p.rope_cs = h->rope_cs;
  // the tile engine's buffers, each at least as large as this schedule needs
  p.x = reinterpret_cast<float*>(scratch + L.x1);
  p.a_o = reinterpret_cast<uint16_t*>(scratch + L.a1[2]);
  p.acc_qkv[0] = reinterpret_cast<float*>(scratch + L.acc1_qkv);
  p.acc_qkv[1] = reinterpret_cast<float*>(scratch + L.acc_qkv_b);
  p.acc_gu = reinterpret_cast<float*>(scratch + L.acc1_gu);
  p.logits = reinterpret_cast<float*>(scratch + L.logits);
  p.kv = reinterpret_cast<uint16_t*>(scratch + L.kv);
  p.Bmax = bmax;
  p.done = reinterpret_cast<unsigned*>(sync + S.done);
  p.qkv_tile = reinterpret_cast<unsigned*>(sync + S.qkv_tile);
  p.att = reinterpret_cast<unsigned*>(sync + S.att);
  p.prep = reinterpret_cast<unsigned*>(sync + S.prep);
  p.decided = reinterpret_cast<unsigned*>(sync + S.decided);
  p.in_code = reinterpret_cast<int32_t*>(sync + S.in_code);
  p.rexp = reinterpret_cast<int*>(sync + S.rexp);
  p.proj_in = g.code_embed_dim != g.hidden;
  p.abort_flag = reinterpret_cast<int*>(sync + S.abort_flag);
  p.status = h->status;
  p.spin_limit = h->wait_ticks > 0 ? h->wait_ticks : kSpinLimit;
  p.withhold = h->withhold_gemm;
  p.NGEMM = S.NGEMM; p.NHT = S.NHT;
  p.trace = h->trace; p.trace_n = h->trace_phases;
  p.B = a.B; p.H = a.H; p.q0 = a.q0; p.out_codes = a.out_codes; p.out_logits = a.out_logits; p.forced = a.forced;
  p.temperature = a.temperature; p.top_k = a.top_k; p.gumbel = a.gumbel;
  p.mode = SM_RUN; p.k_first = 1; p.n_run = g.n_steps; p.n_groups = 1; p.group_rows = a.B;
}

constexpr int kSmMaxDevices = 64;
// Per device: the kernel's shared-memory limit has been set (atomic: first
// calls from several host threads may race to set it, an idempotent call).
std::atomic<bool> g_sm_attr[kSmMaxDevices];

qp_status sm_launch(const qp_handle* h, const SParams& p, uint8_t* sync, size_t sync_bytes, cudaStream_t s) {
  const int dev = h->device;
  std::atomic<bool> local(false);
  std::atomic<bool>* attr = dev >= 0 && dev < kSmMaxDevices ? &g_sm_attr[dev] : &local;
  const size_t smem = kSmOffMisc + sizeof(SMisc) + 1024;
  if (!attr->load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(SM_KERNEL, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess) {
      cudaGetLastError();
      return QP_ERR_CUDA;
    }
    attr->store(true, std::memory_order_release);
  }
  if (cudaMemsetAsync(sync, 0, sync_bytes, s) != cudaSuccess) {
    cudaGetLastError();
    return QP_ERR_CUDA;
  }
  SParams pc = p;
  void* args[] = {&pc};
  if (cudaLaunchCooperativeKernel(reinterpret_cast<void*>(SM_KERNEL), dim3(h->num_sms), dim3(kSmThreads), args,
                                  smem, s) != cudaSuccess) {
    cudaGetLastError();
    return QP_ERR_CUDA;
  }
  return QP_OK;
}

}  // namespace

#if !QP_SMALL_SLOTS && !QP_SMALL_SAMPLED

size_t small_smem_bytes() { return kSmOffMisc + sizeof(SMisc) + 1024; }

bool small_supported(const qp_handle* h, const RunArgs& a) {
  // Q8_0 matrices are served through their f16 hi and lo images (loaded beside them)
  if (h->wfmt == WF_Q8_0 && !h->layer[0].qkv.w16[0]) return false;
  if (a.B < 1 || a.B > kSmallMaxFrames) return false;
  if (a.temperature > 0.f && h->g.vocab > kMaxVocab) return false;
  return true;
}

qp_status run_frames_small(qp_handle* h, const RunArgs& a, uint8_t* scratch, const Scratch& L, int bmax,
                           cudaStream_t s) {
  if (!small_supported(h, a) || a.B > bmax) return QP_ERR_ARG;
  if (a.temperature > 0.f) return run_frames_small_sampled(h, a, scratch, L, bmax, s);
  const SmSync S = sm_sync_layout(h->g, a.B);
  if (L.total - L.sync < S.total) return QP_ERR_ARG;
  uint8_t* sync = scratch + L.sync;
  SParams p{};
  sm_fill(p, h, a, scratch, L, sync, S, bmax);
  return sm_launch(h, p, sync, S.total, s);
}

#elif QP_SMALL_SAMPLED && !QP_SMALL_SLOTS   // the sampling frame-loop kernel

qp_status run_frames_small_sampled(qp_handle* h, const RunArgs& a, uint8_t* scratch, const Scratch& L, int bmax,
                                   cudaStream_t s) {
  const SmSync S = sm_sync_layout(h->g, a.B);
  if (L.total - L.sync < S.total) return QP_ERR_ARG;
  uint8_t* sync = scratch + L.sync;
  SParams p{};
  sm_fill(p, h, a, scratch, L, sync, S, bmax);
  return sm_launch(h, p, sync, S.total, s);
}

#else   // the state-slot kernels, greedy (k_slots_small) and sampling (k_slots_small_sampled)

#if QP_SMALL_SAMPLED
qp_status run_slots_small_sampled(qp_handle* h, const SlotArgs& sa, uint8_t* scratch, const Scratch& L, int bmax,
                                  cudaStream_t s) {
#else
qp_status run_slots_small(qp_handle* h, const SlotArgs& sa, uint8_t* scratch, const Scratch& L, int bmax,
                          cudaStream_t s) {
  if (sa.temperature > 0.f) return run_slots_small_sampled(h, sa, scratch, L, bmax, s);
#endif
  const qp_geometry& g = h->g;
  const int B = sa.B;
  if (B < 1 || B > kSmallMaxFrames || B > bmax) return QP_ERR_ARG;
  RunArgs a{};
  a.B = B; a.H = sa.H; a.q0 = sa.q0; a.out_codes = sa.out_codes; a.out_logits = sa.out_logits;
  a.temperature = sa.temperature; a.top_k = sa.top_k; a.gumbel = sa.gumbel;
  SParams p{};
  // rows in step order (a stable sort keeps the caller's order within a step)
  int order[kSmallMaxFrames];
  int n_groups = 1, group_rows = B;
  for (int b = 0; b < B; ++b) order[b] = b;
  if (sa.mode == SM_STEP) {
    std::stable_sort(order, order + B, [&](int x, int y) { return sa.steps[x] < sa.steps[y]; });
    n_groups = 0;
    group_rows = 0;
    for (int b = 0; b < B; ++b) {
      const int st = sa.steps[order[b]];
      if (b == 0 || st != sa.steps[order[b - 1]]) {
        p.group_start[n_groups] = b;
        p.group_step[n_groups] = st;
        ++n_groups;
      }
    }
    p.group_start[n_groups] = B;
    for (int i = 0; i < n_groups; ++i) group_rows = std::max(group_rows, p.group_start[i + 1] - p.group_start[i]);
  }
  for (int b = 0; b < B; ++b) {
    p.row_perm[b] = order[b];
    p.row_slot[b] = sa.slots[order[b]];
    p.row_step[b] = sa.mode == SM_STEP ? sa.steps[order[b]] : 1;
  }
  const SmSync S = sm_sync_layout(g, B, sa.mode);
  if (L.total - L.sync < S.total) return QP_ERR_ARG;
  uint8_t* sync = scratch + L.sync;
  sm_fill(p, h, a, scratch, L, sync, S, bmax);
  p.mode = sa.mode;
  p.k_first = sa.mode == SM_STEP ? 2 : 1;
  p.n_run = 1;
  p.n_groups = n_groups;
  p.group_rows = group_rows;
  p.code_in = sa.codes_in;
  return sm_launch(h, p, sync, S.total, s);
}

#endif

}  // namespace qp
