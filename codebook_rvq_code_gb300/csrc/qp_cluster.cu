// The Code Predictor frame loop for small batches on thread-block clusters:
// one persistent kernel of 8-CTA clusters, scheduled so that most of a
// layer's dependencies resolve inside a cluster.
//
// It computes what the other two schedules compute (the whole greedy frame
// loop as one fixed GPU program over a preallocated KV cache for the short
// bounded context: "テキスト音声合成モデルを50ミリ秒未満で応答させる方法",
// section "Qwen3-TTSの最適化方法", item 3).  What differs is where partial
// products meet.  A layer is two cluster jobs:
//
//   * attention, one cluster per kv head j: its 8 CTAs multiply the group's
//     512 q|k|v weight rows (q heads 2j and 2j+1, k head j, v head j: four
//     128-row tiles) by the normalised input, CTA r taking tile r/2 over
//     half r%2 of K.  Each drain stores its partial products, by
//     asynchronous stores counted on the receiver's mbarrier, into the
//     receive buffer of the CTA that owns the frame (frame b: CTA b mod 8),
//     which adds the two halves, runs the frame's attention over the KV cache
//     it keeps in its tensor memory and stores the frame's output row into
//     every peer's operand of the O projection.  CTA r multiplies O's
//     128-row tile r over the group's 256 columns and adds the result into
//     the residual stream;
//   * MLP, one cluster per 256 columns of the FFN: the gate and up tiles of
//     those columns split the same way, SwiGLU from the peers' partials into
//     every peer's down-projection operand, CTA r adds down's tile r over
//     the 256 columns into the residual stream;
//   * the head, one cluster per 512 logits (four tiles, two K halves): each
//     CTA completes 64 logits per frame from its own and its partner's
//     halves, writes them out if asked and folds their argmax into the
//     frame's decision word with one 64-bit atomic max.
//
// An operand row is f16(x * w_norm * 2^-e), e from the mean square of the
// CTA's K half of the row; the drain applies 2^e / RMS, the exact RMS
// following from this half's sum of squares and the partner's, which
// arrives while the MMAs run.  The only grid-wide dependencies are the
// residual stream after O and after down (counters in global memory, as in
// the other schedules) and the step's decisions; inside a cluster every
// exchange is an asynchronous store into a peer's shared memory, counted in
// bytes on the peer's mbarrier.  Step 1's projection is spread over all CTAs
// (partials added into the residual stream, each unit scaling its H slice
// into f16's range by a power of two).
//
// Roles per CTA: warps 0-7 consume (operand builds, drains, attention,
// SwiGLU, decisions), warp 8 streams weights, warp 9 issues the MMAs.  Every
// wait is bounded and honours the grid-wide abort flag; no CTA leaves before
// its whole cluster is done with its shared memory.
#include <algorithm>
#include <atomic>
#include <cstdlib>

#include "qp_device.cuh"

namespace qp {

namespace {

constexpr int kCl = 8;                        // CTAs per cluster
constexpr int kClConsWarps = 8;
constexpr int kClCons = kClConsWarps * 32;
constexpr int kClProdWarp = 8;
constexpr int kClMmaWarp = 9;
constexpr int kClThreads = 10 * 32;
constexpr int kClMaxRows = 64;                // activation rows of one GEMM (2B at step 1)
constexpr int kClHold = 8;                    // input chunks a consumer thread keeps in registers
constexpr int kClSplitRows = 24;              // from this many rows the four CTAs of a K half share the loads

constexpr uint32_t kClWSlot = kTileM * kKs * 2;       // one 128 x 128 f16 weight slice
// Weight ring slots.  Four hold a whole QKV, gate/up or head task (measured:
// 116.6 us per step at one frame and 154.1 at 32, against 120.5 and 155.6
// with five).
constexpr int kClNW = 4;
// the 16-bit MMA loop waits for all of a task's slices (up to four) before its first MMA
static_assert(kClNW >= 4, "a 16-bit task's weight slices must all fit the ring");
constexpr uint32_t kClOffW = 0;
constexpr uint32_t kClOffOp = kClNW * kClWSlot;       // operand region (K half; then the partials)
constexpr uint32_t kClOpBytes = 65536;
constexpr uint32_t kClOffOp2 = kClOffOp + 32768;      // O / down operand (second half of the region)
// Partial products pushed here by the peers: an attention CTA's frames (q|k|v
// tiles x K halves), or a SwiGLU CTA's 32 columns of gate and up.
constexpr uint32_t kClOffRecv = kClOffOp + kClOpBytes;
constexpr uint32_t kClRecvBytes = 32768;
constexpr uint32_t kClOffMisc = kClOffRecv + kClRecvBytes;
// Tensor memory: the accumulator (up to 64 columns), then the KV cache of
// the frames this CTA runs attention for.  Lane quarter q holds frame
// r + 8q; per layer 64 columns: k of positions 0..15 in columns 2t, 2t + 1
// (f16, dims 4l..4l+3 in lane l of the quarter), v in 32 + 2t, 33 + 2t.
constexpr uint32_t kClTmemCols = 512;
constexpr uint32_t kClKvCol = 64;
constexpr uint32_t kClKvColsPerLayer = 4 * kMaxCtx;
constexpr int kClMaxLayers = int((kClTmemCols - kClKvCol) / kClKvColsPerLayer);
static_assert(kMaxCtx == 16, "the TMEM cache holds 16 positions per layer");
static_assert(kClusterMaxFrames <= 4 * kCl, "one frame per lane quarter of each CTA");
static_assert(kClusterMaxFrames <= kCl * kClConsWarps / 2, "attention: one (frame, q head) per warp");

enum { CBAR_CONS = 1 };
enum { T_PROJ = 0, T_QKV, T_O, T_GU, T_DOWN, T_HEAD };

struct CMisc {
  uint64_t wfull[kClNW], wempty[kClNW];
  uint64_t opfull, accfull, mmadone;
  uint64_t opx;                  // the O or down operand's rows, written by the peers, have landed
  uint64_t prx;                  // the partial products this CTA consumes have landed
  uint64_t psx;                  // the partner's sums of squares have landed (split: the rows' statistics)
  uint64_t nx;                   // split: the normalised operand's rows, written by the half's four CTAs, have landed
  uint32_t tmem_base;
  int flag[2];                   // a wait's outcome for all consumers (alternating: a fast thread's next
                                 // wait may write before a slow one has read the last)
  float ssw[kClConsWarps][kClMaxRows / 4];   // per-warp partial sums of squares of one pass's rows
  float ssx[kClMaxRows];         // per row: this K half's sum of squares (split: a peer's row stored by its builder)
  float ssp[kClMaxRows];         // per row: the other K half's, stored by the partner (split: by the row's builder)
  float inv[kClMaxRows];         // per row: the factor a drain applies (2^e / RMS, or 2^e for the projection)
  float rsc[kClMaxRows];         // per row: 2^-e, the operand's range scale (split: as ssx)
  int code[kClMaxRows];          // step k >= 2: the code each frame's input embeds
};

// dynamic shared memory (with 1 KB for aligning its base) within the 227 KB a CTA may use
static_assert(kClOffMisc + sizeof(CMisc) + 1024 <= 227 * 1024, "shared memory layout too large");

struct CLayer {
  const uint16_t* w[4];    // qkv, o, gu, down: tile-packed f16 (qp_weights.cu); a Q8_0 matrix's hi image
  const uint16_t* wl[4];   // Q8_0 matrices: the lo image (hi + lo = d * q), else null
  const float* attn_norm; const float* q_norm; const float* k_norm; const float* ffn_norm;
};

struct CParams {
  int d, qw, kvw, F, V, th, L, n_kv, n_steps, q0_vocab;
  float eps;
  bool embed_f16;
  const uint16_t* w_proj; const uint16_t* w_proj_lo; const float* b_proj; const uint16_t* e0;
  bool proj_in;            // Talker-wide code tables: each step's input row is projected (a GEMM per step)
  CLayer layer[kMaxLayers];
  const float* out_norm;
  const uint16_t* embed[kMaxSteps];
  const uint16_t* w_head[kMaxSteps];
  const uint16_t* w_head_lo[kMaxSteps];   // Q8_0 heads: the lo images, else null
  const float2* rope_cs;
  // scratch
  float* x;                // residual streams [step][2B][d], zeroed per call
  unsigned* proj_done;     // [step]: projection units finished (step 1; every step with Talker-wide tables)
  unsigned* att_done;      // [step][layer]: attention CTAs finished (O added)
  unsigned* mlp_done;      // [step][layer]: MLP CTAs finished (down added)
  unsigned* head_done;     // [step]: head CTAs finished (decisions folded in)
  unsigned long long* best;   // [step][frame]: packed (logit, index) maximum
  int* abort_flag; int* status;
  long long spin_limit;
  int withhold;            // testing (qp_debug.h): >= 0 makes CTA 0 skip its first attention count
  unsigned long long* trace; int trace_n;   // event log (qp_debug.h), or null
  // jobs
  int n_cl;                // clusters in the grid
  int n_att, n_mlp, n_head, n_proj;   // jobs of each kind (projection: units over all CTAs)
  // call
  int B;
  const float* H; const int32_t* q0; int32_t* out_codes; float* out_logits; const int32_t* forced;
};

// ------------------------------------------------------------ cluster PTX
__device__ __forceinline__ uint32_t cl_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cl_map(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}
__device__ __forceinline__ bool cl_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Asynchronous store into a peer's shared memory, counted in bytes on the
// peer's mbarrier at cluster address `bar`.
__device__ __forceinline__ void cl_st2_async(uint32_t a, uint2 v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];" ::"r"(a),
               "r"(v.x), "r"(v.y), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void cl_st4u_async(uint32_t a, uint4 v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(a),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void cl_st1_async(uint32_t a, float v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(a), "f"(v), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void cl_st4_async(uint32_t a, float4 v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(a),
               "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar)
               : "memory");
}
// Hardware barrier of every thread of the cluster.
__device__ __forceinline__ void cl_barrier_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ------------------------------------------------------------ tracing
// Per-CTA event log after the section stamps: consumer events in [0, 8192),
// MMA-warp events in [8192, 16384); one word = (globaltimer ns mod 2^48) <<
// 16 | code << 12 | task index.  Compiled in only with QP_TRACE.
enum {
  CEV_START = 1, CEV_READY = 2, CEV_SSYNC = 3, CEV_OPREADY = 4, CEV_ACC = 5, CEV_S1 = 6, CEV_WORK = 7,
  CEV_S3 = 8, CEV_PUB = 9, CEV_WWAIT = 10, CEV_WREADY = 11, CEV_COMMIT = 12, CEV_MOP = 13, CEV_SUB = 14,
  CEV_BSUB = 15
};
#ifdef QP_TRACE
__device__ __forceinline__ void cl_ev(const CParams& p, unsigned& idx, int base, int code, int task) {
  if (p.trace && idx < 8192) {
    unsigned long long* b = p.trace + size_t(p.trace_n) * gridDim.x * 2 + size_t(blockIdx.x) * 16384 + base;
    b[idx++] = ((globaltimer_ns() & 0xFFFFFFFFFFFFull) << 16) | (unsigned long long)(code & 15) << 12 |
               unsigned(task & 4095);
  }
}
#else
__device__ __forceinline__ void cl_ev(const CParams&, unsigned&, int, int, int) {}
#endif

// --------------------------------------------------------------- program
// A CTA's tasks, in the order every role walks them.  Per step k: step 1's
// projection units, then per layer this cluster's attention jobs (a QKV and
// an O task each) and MLP jobs (gate/up and down), then its head jobs.
struct Task {
  int kind, k, l, job;
};
// Jobs of each kind are dealt to clusters round-robin; MLP jobs from the
// last cluster down, so that clusters with an attention job take fewer.
__device__ __forceinline__ int n_mine(int n_jobs, int n_cl, int c) { return c < n_jobs % n_cl ? n_jobs / n_cl + 1 : n_jobs / n_cl; }
__device__ __forceinline__ int cl_proj_units(const CParams& p) {
  const int g = blockIdx.x, G = gridDim.x;
  return g < p.n_proj ? (p.n_proj - 1 - g) / G + 1 : 0;
}
struct Prog {
  int c, na, nm, nh, np, per_layer, rest;   // rest: a step's tasks after its projection units
};
__device__ __forceinline__ Prog cl_prog(const CParams& p) {
  Prog g;
  g.c = int(blockIdx.x) / kCl;
  g.na = n_mine(p.n_att, p.n_cl, g.c);
  g.nm = n_mine(p.n_mlp, p.n_cl, p.n_cl - 1 - g.c);
  g.nh = n_mine(p.n_head, p.n_cl, g.c);
  g.np = cl_proj_units(p);
  g.per_layer = 2 * (g.na + g.nm);
  g.rest = p.L * g.per_layer + g.nh;
  return g;
}
// EXT: the kernel instantiation that serves Q8_0 matrices (their hi and lo
// images) and Talker-wide code tables (a projection GEMM per step); the
// other one keeps the smaller code of 16-bit weights and unprojected tables.
template <bool EXT>
__device__ __forceinline__ bool cl_proj_in(const CParams& p) { return EXT && p.proj_in; }
// Projection units of step k's inputs: step 1 always, later steps with Talker-wide tables.
template <bool EXT>
__device__ __forceinline__ int cl_step_proj(const CParams& p, const Prog& g, int k) {
  return (k == 1 || cl_proj_in<EXT>(p)) ? g.np : 0;
}
template <bool EXT>
__device__ __forceinline__ int cl_n_tasks(const CParams& p, const Prog& g) {
  return g.np + g.rest + (p.n_steps - 1) * (cl_step_proj<EXT>(p, g, 2) + g.rest);
}
template <bool EXT>
__device__ Task cl_task(const CParams& p, const Prog& g, int i) {
  Task t{};
  const int first = g.np + g.rest;
  if (i < first) {
    t.k = 1;
  } else {
    i -= first;
    const int ps = cl_step_proj<EXT>(p, g, 2) + g.rest;
    t.k = 2 + i / ps;
    i %= ps;
  }
  const int pk = cl_step_proj<EXT>(p, g, t.k);
  if (i < pk) {
    t.kind = T_PROJ; t.l = 0; t.job = int(blockIdx.x) + i * int(gridDim.x);
    return t;
  }
  i -= pk;
  if (i >= p.L * g.per_layer) {
    t.kind = T_HEAD; t.l = p.L; t.job = g.c + (i - p.L * g.per_layer) * p.n_cl;
    return t;
  }
  t.l = i / g.per_layer;
  i %= g.per_layer;
  if (i < 2 * g.na) {
    t.kind = (i & 1) ? T_O : T_QKV;
    t.job = g.c + (i >> 1) * p.n_cl;
  } else {
    i -= 2 * g.na;
    t.kind = (i & 1) ? T_DOWN : T_GU;
    t.job = (p.n_cl - 1 - g.c) + (i >> 1) * p.n_cl;
  }
  return t;
}

// Activation rows of a task's GEMM.
__device__ __forceinline__ int cl_rows(const CParams& p, const Task& t) {
  if (t.kind == T_HEAD) return p.B;
  return t.k == 1 ? 2 * p.B : p.B;
}
__device__ __forceinline__ int cl_npad(int R) { return (R + 15) & ~15; }
// The MMA of a task: its weight slices (0 = none: an O or down task whose
// tile this CTA does not have).
__device__ __forceinline__ int cl_nsl(const CParams& p, const Task& t) {
  const int r = int(cl_rank());
  switch (t.kind) {
    case T_PROJ: return 1;
    case T_O: case T_DOWN: return r < p.d / kTileM ? 2 : 0;
    default: return p.d / 256;
  }
}
// Images of each weight slice of the task: 2 for a Q8_0 matrix (hi, lo), else 1.
template <bool EXT>
__device__ __forceinline__ int cl_nimg(const CParams& p, const Task& t) {
  if (!EXT) return 1;
  switch (t.kind) {
    case T_PROJ: return p.w_proj_lo ? 2 : 1;
    case T_HEAD: return p.w_head_lo[t.k - 1] ? 2 : 1;
    case T_QKV: return p.layer[t.l].wl[0] ? 2 : 1;
    case T_O: return p.layer[t.l].wl[1] ? 2 : 1;
    case T_GU: return p.layer[t.l].wl[2] ? 2 : 1;
    default: return p.layer[t.l].wl[3] ? 2 : 1;
  }
}
// Weight slice s of the task's unit, image img: tile `mt` of the matrix, K slice `ks`.
__device__ __forceinline__ const uint8_t* cl_slice(const CParams& p, const Task& t, int s, int img) {
  const int r = int(cl_rank()), tq = r >> 1, h = r & 1, nkh = p.d / 256;
  const uint16_t* w;
  int mt, ks, K;
  switch (t.kind) {
    case T_PROJ: {
      const int nks = p.th / kKs;
      w = img ? p.w_proj_lo : p.w_proj; K = p.th; mt = t.job / nks; ks = t.job % nks;
      break;
    }
    case T_QKV: {
      const int j = t.job;
      const int tiles[4] = {2 * j, 2 * j + 1, p.qw / kTileM + j, (p.qw + p.kvw) / kTileM + j};
      w = img ? p.layer[t.l].wl[0] : p.layer[t.l].w[0]; K = p.d; mt = tiles[tq]; ks = h * nkh + s;
      break;
    }
    case T_O:
      w = img ? p.layer[t.l].wl[1] : p.layer[t.l].w[1]; K = p.qw; mt = r; ks = 2 * t.job + s;
      break;
    case T_GU: {
      const int m = t.job, fq = p.F / kTileM;
      const int tiles[4] = {2 * m, 2 * m + 1, fq + 2 * m, fq + 2 * m + 1};
      w = img ? p.layer[t.l].wl[2] : p.layer[t.l].w[2]; K = p.d; mt = tiles[tq]; ks = h * nkh + s;
      break;
    }
    case T_DOWN:
      w = img ? p.layer[t.l].wl[3] : p.layer[t.l].w[3]; K = p.F; mt = r; ks = 2 * t.job + s;
      break;
    default:   // T_HEAD
      w = img ? p.w_head_lo[t.k - 1] : p.w_head[t.k - 1]; K = p.d; mt = 4 * t.job + tq; ks = h * nkh + s;
      break;
  }
  return reinterpret_cast<const uint8_t*>(w) + (size_t(mt) * K * kTileM + size_t(ks) * kTileM * kKs) * 2;
}
// Operand slice s of the task in shared memory.
__device__ __forceinline__ uint32_t cl_op_off(const Task& t, int s, uint32_t opsz) {
  return ((t.kind == T_O || t.kind == T_DOWN) ? kClOffOp2 : kClOffOp) + uint32_t(s) * opsz;
}

// ---------------------------------------------------------------- producer
template <bool EXT>
__device__ void cl_producer(const CParams& p, CMisc& ms, uint8_t* smem) {
  const uint64_t pol = policy_evict_first();
  const Prog g = cl_prog(p);
  const int n = cl_n_tasks<EXT>(p, g);
  uint32_t it = 0;
  for (int i = 0; i < n; ++i) {
    const Task t = cl_task<EXT>(p, g, i);
    const int nsl = cl_nsl(p, t), nimg = cl_nimg<EXT>(p, t);
    for (int s = 0; s < nsl; ++s) {
      for (int img = 0; img < nimg; ++img) {
        const uint32_t slot = it % kClNW, u = it / kClNW;
        if (u > 0 && !mwait(p, &ms.wempty[slot], (u - 1) & 1)) goto drain;
        mbar_expect_tx(&ms.wfull[slot], kClWSlot);
        bulk_g2s_stream(smem + kClOffW + slot * kClWSlot, cl_slice(p, t, s, img), kClWSlot, &ms.wfull[slot], pol);
        ++it;
      }
    }
  }
drain:
  for (uint32_t k = it > uint32_t(kClNW) ? it - kClNW : 0; k < it; ++k) mbar_wait(&ms.wfull[k % kClNW], (k / kClNW) & 1);
}

// --------------------------------------------------------------- MMA warp
__device__ bool cl_wait_slot(const CParams& p, CMisc& ms, uint32_t w, unsigned& evi, int i) {
  if (mbar_try_wait(&ms.wfull[w % kClNW], (w / kClNW) & 1)) {
    cl_ev(p, evi, 8192, CEV_WREADY, i);
    return true;
  }
  if (!mwait(p, &ms.wfull[w % kClNW], (w / kClNW) & 1)) return false;
  cl_ev(p, evi, 8192, CEV_WWAIT, i);
  return true;
}

template <bool SPLIT, bool EXT>
__device__ void cl_mma(const CParams& p, CMisc& ms, uint8_t* smem) {
  const Prog g = cl_prog(p);
  const int n = cl_n_tasks<EXT>(p, g);
  uint32_t wit = 0, opw = 0, xseq = 0, nseq = 0;   // weight slots; phases of opfull, opx and nx waited for
  unsigned evi = 0;
  for (int i = 0; i < n; ++i) {
    const Task t = cl_task<EXT>(p, g, i);
    const int nsl = cl_nsl(p, t), nimg = cl_nimg<EXT>(p, t);
    if (nsl == 0) continue;
    const int np = cl_npad(cl_rows(p, t));
    const uint32_t idesc = idesc_f16(kTileM, np);
    const uint32_t blb = uint32_t(np / 8) * 128, opsz = uint32_t(np) * kKs * 2;
    // the task's weight slices first (usually there long before the operand):
    // a wait between MMAs stalls the issuing thread while the tensor pipe
    // drains.  A task with more slices than the ring holds (Q8_0 images) waits
    // for the rest as it goes.
    const int nw = nsl * nimg, pre = nw <= kClNW ? nw : 0;
    for (int s = 0; s < pre; ++s)
      if (!cl_wait_slot(p, ms, wit + uint32_t(s), evi, i)) goto out;
    if (t.kind == T_O || t.kind == T_DOWN) {
      // the peers' asynchronous stores of the operand's rows, counted on opx
      if (!mwait(p, &ms.opx, xseq & 1)) goto out;
      ++xseq;
      fence_proxy_async_shared();   // those generic-proxy writes, for the tensor cores' reads
    } else if (SPLIT && t.kind != T_PROJ && cl_rows(p, t) >= kClSplitRows) {
      // a normalised operand built by the half's four CTAs, counted on nx
      if (!mwait(p, &ms.nx, nseq & 1)) goto out;
      ++nseq;
      fence_proxy_async_shared();
    } else {
      if (!mwait(p, &ms.opfull, opw & 1)) goto out;
      ++opw;
    }
    cl_ev(p, evi, 8192, CEV_MOP, i);
    tc_fence_after();
    if (!EXT) {   // one image per slice, all of them already waited for
      for (int s = 0; s < nsl; ++s) {
        const uint32_t ws = wit % kClNW;
        const uint32_t a0 = smem_u32(smem + kClOffW + ws * kClWSlot);
        const uint32_t b0 = smem_u32(smem + cl_op_off(t, s, opsz));
#pragma unroll
        for (int j = 0; j < kKs / 16; ++j) {
          const uint64_t ad = smem_desc(a0 + uint32_t(j) * 2 * (kTileM / 8) * 128, (kTileM / 8) * 128, 128);
          const uint64_t bd = smem_desc(b0 + uint32_t(j) * 2 * blb, blb, 128);
          mma_f16(ms.tmem_base, ad, bd, idesc, (s == 0 && j == 0) ? 0u : 1u);
        }
        mma_commit(&ms.wempty[ws]);
        ++wit;
      }
    } else
    for (int s = 0; s < nsl; ++s) {
      const uint32_t b0 = smem_u32(smem + cl_op_off(t, s, opsz));
      for (int img = 0; img < nimg; ++img) {
        const uint32_t ws = wit % kClNW;
        if (!pre) {
          if (!cl_wait_slot(p, ms, wit, evi, i)) goto out;
          tc_fence_after();
        }
        const uint32_t a0 = smem_u32(smem + kClOffW + ws * kClWSlot);
#pragma unroll
        for (int j = 0; j < kKs / 16; ++j) {
          const uint64_t ad = smem_desc(a0 + uint32_t(j) * 2 * (kTileM / 8) * 128, (kTileM / 8) * 128, 128);
          const uint64_t bd = smem_desc(b0 + uint32_t(j) * 2 * blb, blb, 128);
          mma_f16(ms.tmem_base, ad, bd, idesc, (s == 0 && img == 0 && j == 0) ? 0u : 1u);
        }
        mma_commit(&ms.wempty[ws]);
        ++wit;
      }
    }
    mma_commit(&ms.accfull);
    cl_ev(p, evi, 8192, CEV_COMMIT, i);
  }
out:
  mma_commit(&ms.mmadone);
  mbar_wait(&ms.mmadone, 0);
}

// ------------------------------------------------------ consumer helpers
struct CState {
  uint32_t opseq;   // tasks whose MMA ran
  uint32_t fseq;    // waits whose outcome went through ms.flag
  uint32_t rseq;    // phases of ms.prx
  uint32_t pseq;    // phases of ms.psx
  int r;            // rank in the cluster
  int task;         // the task in progress (event log)
  unsigned evi;     // events logged (thread 0)
};
__device__ __forceinline__ void cev(const CParams& p, CState& st, int code) {
  if (threadIdx.x == 0) cl_ev(p, st.evi, 0, code, st.task);
}

// Bounded wait for a phase of an mbarrier that peers complete (acquire at
// cluster scope).
template <class Par>
__device__ bool cl_mwait(const Par& p, uint64_t* bar, uint32_t parity) {
  if (cl_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (unsigned it = 1;; ++it) {
    if (cl_try_wait(bar, parity)) return true;
    if ((it & 255) == 0) {
      if (aborted(p)) return false;
      if (clock64() - t0 > p.spin_limit) { abort_all(p); return false; }
    }
  }
}
// One thread waits on a global counter; the consumers meet and read after.
__device__ bool cl_wait_ctr(const CParams& p, CMisc& ms, CState& st, const unsigned* ctr, unsigned want) {
  int* f = &ms.flag[st.fseq++ & 1];
  if (threadIdx.x == 0) *f = poll_geq(p, ctr, want);
  cev(p, st, CEV_READY);
  named_bar(CBAR_CONS, kClCons);
  return *f != 0;
}
__device__ bool cl_wait_acc(const CParams& p, CMisc& ms, CState& st) {
  int* f = &ms.flag[st.fseq++ & 1];
  if (threadIdx.x == 0) *f = mwait(p, &ms.accfull, st.opseq & 1);
  cev(p, st, CEV_ACC);
  named_bar(CBAR_CONS, kClCons);
  ++st.opseq;
  tc_fence_after();
  return *f != 0;
}
// The operand is complete in shared memory: hand it to the MMA warp.
__device__ __forceinline__ void cl_op_ready(const CParams& p, CMisc& ms, CState& st) {
  fence_proxy_async_shared();
  named_bar(CBAR_CONS, kClCons);
  if (threadIdx.x == 0) mbar_arrive(&ms.opfull);
  cev(p, st, CEV_OPREADY);
}
// Publish this CTA's count on `ctr` after every consumer's global writes.
__device__ __forceinline__ void cl_publish(const CParams& p, CState& st, unsigned* ctr) {
  named_bar(CBAR_CONS, kClCons);
  if (threadIdx.x == 0) {
    fence_acq_rel_gpu();
    red_relaxed_add(ctr, 1u);
  }
  cev(p, st, CEV_PUB);
}

// RMSNorm of two 128-vectors held as 4 values per lane (a frame's k and its
// q head) with their norms' weights (this lane's four), then rotate-half
// RoPE with this lane's factors c (pairs (i, i+64) sit in lanes l and l^16);
// the two warp reductions interleave, so their shuffle latencies overlap.
__device__ __forceinline__ void norm_rope_w2(float4 xa, float4 wa, float4 xb, float4 wb, const float2 (&c)[4],
                                             float eps, int lane, float4& oa, float4& ob) {
  float sa = xa.x * xa.x + xa.y * xa.y + xa.z * xa.z + xa.w * xa.w;
  float sb = xb.x * xb.x + xb.y * xb.y + xb.z * xb.z + xb.w * xb.w;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sa += __shfl_xor_sync(0xffffffffu, sa, o);
    sb += __shfl_xor_sync(0xffffffffu, sb, o);
  }
  const float ra = rsqrtf(sa / 128.f + eps), rb = rsqrtf(sb / 128.f + eps);
  const float va[4] = {xa.x * ra * wa.x, xa.y * ra * wa.y, xa.z * ra * wa.z, xa.w * ra * wa.w};
  const float vb[4] = {xb.x * rb * wb.x, xb.y * rb * wb.y, xb.z * rb * wb.z, xb.w * rb * wb.w};
  float a[4], b[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float pa = __shfl_xor_sync(0xffffffffu, va[e], 16), pb = __shfl_xor_sync(0xffffffffu, vb[e], 16);
    a[e] = lane < 16 ? va[e] * c[e].x - pa * c[e].y : va[e] * c[e].x + pa * c[e].y;
    b[e] = lane < 16 ? vb[e] * c[e].x - pb * c[e].y : vb[e] * c[e].x + pb * c[e].y;
  }
  oa = make_float4(a[0], a[1], a[2], a[3]);
  ob = make_float4(b[0], b[1], b[2], b[3]);
}

// L2 loads issued where they stand (volatile: the compiler keeps them ahead
// of the barriers that follow, so their latency overlaps the wait).
__device__ __forceinline__ float4 ldv_f4(const void* src) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(src));
  return v;
}
// 32 lanes x 32 columns of 32-bit words from TMEM, issued only: tmem_wait_ld2
// completes them.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// Wait for this thread's TMEM loads; the registers pass through the wait so
// that no use of them is scheduled ahead of it.
__device__ __forceinline__ void tmem_regs_after_wait(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_wait_ld2(uint32_t (&a)[32], uint32_t (&b)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  tmem_regs_after_wait(a);
  tmem_regs_after_wait(b);
}
// Two 32-bit words into columns taddr, taddr + 1 of this thread's lane.
__device__ __forceinline__ void tmem_st2(uint32_t taddr, uint2 v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1, %2};" ::"r"(taddr), "r"(v.x), "r"(v.y) : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void ld8f(const float* src, float (&v)[8]) {
  const float4 a = ldv_f4(src), b = ldv_f4(src + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void ld8e(const uint16_t* src, bool f16, float (&v)[8]) {
  const uint4 e = __ldg(reinterpret_cast<const uint4*>(src));
  const uint32_t w[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) { v[2 * i] = e16_to_f32(w[i], f16); v[2 * i + 1] = e16_to_f32(w[i] >> 16, f16); }
}
__device__ __forceinline__ uint4 pack8h(const float (&v)[8]) {
  const uint2 a = pack4_f16(v[0], v[1], v[2], v[3]), b = pack4_f16(v[4], v[5], v[6], v[7]);
  return make_uint4(a.x, a.y, b.x, b.y);
}
// u16 index of operand element (row n, column k in its 128-column slice),
// the K-major core-matrix image [16 k groups][npad/8][8 rows][8 k].
__device__ __forceinline__ uint32_t op_idx(int n, int k, int n8) {
  return uint32_t(((k >> 3) * n8 + (n >> 3)) * 64 + (n & 7) * 8 + (k & 7));
}

// The 8 input values at column `col` of row n of a normalised GEMM's input:
// the residual row, or at step k >= 2 layer 0 the frame's code embedding.
struct InSrc {
  const float* x;          // residual rows (row stride d), or null
  const uint16_t* emb;     // the step's code table (embedding rows), or null
  int row_mul, row_add;    // residual row = n * row_mul + row_add
};
__device__ __forceinline__ void in_load8(const CParams& p, const CMisc& ms, const InSrc& in, int n, int col,
                                         float (&v)[8]) {
  if (in.emb) ld8e(in.emb + size_t(ms.code[n]) * p.d + col, p.embed_f16, v);
  else ld8f(in.x + size_t(n * in.row_mul + in.row_add) * p.d + col, v);
}

// Build the operand of a normalised GEMM over this CTA's K half: rows
// n < R of input * w_norm * 2^-e, as f16, into slices 0..nkh-1 of the
// operand region, e from the row's mean square over this K half
// (qp_device.cuh, range_exp), and hand it to the MMA warp; the drain applies
// 2^e / RMS to the partial products, the row's 1/RMS following from this
// half's sum of squares and the partner's.
//   * Up to kClSplitRows rows each CTA loads every row of its half, starts
//     the MMAs, and exchanges the sums of squares with its partner by
//     asynchronous stores while they run.
//   * From kClSplitRows rows the four CTAs of a half (ranks h, h+2, h+4,
//     h+6) share the loads: CTA h+2g loads, scales and converts rows n = g
//     (mod 4) and stores them asynchronously into all four operands, counted
//     on each one's ms.nx, which the MMA warp waits for; the rows' sums of
//     squares and scales go the same way to the eight CTAs (ms.psx).
// Thread t takes column chunk t % CH (8 columns) of local rows t / CH + RP i.
template <bool SPLIT>
__device__ bool cl_build_norm(const CParams& p, CMisc& ms, CState& st, uint8_t* smem, const InSrc& in,
                              const float* wn, int R) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int half = p.d / 2, CH = half / 8, RP = kClCons / CH, c = t % CH, h = st.r & 1;
  const bool split = SPLIT && R >= kClSplitRows;
  const int G = split ? 4 : 1, g = split ? st.r >> 1 : 0;
  const int RL = R > g ? (R - g + G - 1) / G : 0;   // this CTA's rows: n = g + G * (local row)
  const int col = h * half + c * 8;   // global column
  const int passes = (RL + RP - 1) / RP;
  const int np = cl_npad(R), n8 = np / 8;
  const uint32_t opsz = uint32_t(np) * kKs * 2;
  // split: all R rows of the half will land in this CTA's operand
  if (split && t == 0) mbar_expect_tx(&ms.nx, uint32_t(R) * uint32_t(p.d));
  // the norm's weights for this thread's 8 columns, in flight with the row loads
  const float4 w0 = __ldg(reinterpret_cast<const float4*>(wn + col));
  const float4 w1 = __ldg(reinterpret_cast<const float4*>(wn + col + 4));
  float hold[kClHold][8];
  // pass 1: sums of squares, the first kClHold chunks kept in registers
  // (their loads all in flight together); a warp's 32 lanes all belong to
  // one row (CH >= 32)
#pragma unroll
  for (int i = 0; i < kClHold; ++i) {
    const int li = t / CH + RP * i;
#pragma unroll
    for (int e = 0; e < 8; ++e) hold[i][e] = 0.f;
    if (i < passes && li < RL) in_load8(p, ms, in, g + G * li, col, hold[i]);
  }
#pragma unroll
  for (int i = 0; i < kClHold; ++i) {
    if (i < passes) {   // warp-uniform
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) ss += hold[i][e] * hold[i][e];
      ss = warp_sum(ss);
      if (lane == 0) ms.ssw[warp][i] = ss;
    }
  }
  cev(p, st, CEV_BSUB);
  for (int i = kClHold; i < passes; ++i) {
    const int li = t / CH + RP * i;
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (li < RL) in_load8(p, ms, in, g + G * li, col, v);
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) ss += v[e] * v[e];
    ss = warp_sum(ss);
    if (lane == 0) ms.ssw[warp][i] = ss;
  }
  named_bar(CBAR_CONS, kClCons);
  if (t < RL) {
    const int slot = t % RP, i = t / RP, w0 = slot * CH / 32, n = g + G * t;
    float s = 0.f;
    for (int w = 0; w < CH / 32; ++w) s += ms.ssw[w0 + w][i];
    const float rs = exp2i(-range_exp(s / float(half)));
    ms.ssx[n] = s;
    ms.rsc[n] = rs;
    if (split) {   // the row's statistics to the other CTAs of both halves, ahead of the MMAs
      const uint32_t xa = smem_u32(&ms.ssx[n]), ra = smem_u32(&ms.rsc[n]), pa = smem_u32(&ms.ssp[n]);
      const uint32_t bar = smem_u32(&ms.psx);
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) {
        const uint32_t mate = uint32_t(h + 2 * gg), other = uint32_t((h ^ 1) + 2 * gg);
        if (gg != g) {
          cl_st1_async(cl_map(xa, mate), s, cl_map(bar, mate));
          cl_st1_async(cl_map(ra, mate), rs, cl_map(bar, mate));
        }
        cl_st1_async(cl_map(pa, other), s, cl_map(bar, other));
      }
    }
  }
  named_bar(CBAR_CONS, kClCons);
  cev(p, st, CEV_BSUB);
  // pass 2: f16(x * w * 2^-e) into the operand slices (of all four CTAs of the half, split)
  const float w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
  const int kl = c * 8, s = kl / kKs, kk = kl % kKs;
  uint16_t* op = reinterpret_cast<uint16_t*>(smem + kClOffOp + uint32_t(s) * opsz);
  auto put = [&](int n, const float (&v)[8]) {
    const uint4 hv = pack8h(v);
    if (!split) {
      *reinterpret_cast<uint4*>(op + op_idx(n, kk, n8)) = hv;
    } else {
      const uint32_t a = smem_u32(op + op_idx(n, kk, n8)), bar = smem_u32(&ms.nx);
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) {
        const uint32_t mate = uint32_t(h + 2 * gg);
        cl_st4u_async(cl_map(a, mate), hv, cl_map(bar, mate));
      }
    }
  };
#pragma unroll
  for (int i = 0; i < kClHold; ++i) {
    const int li = t / CH + RP * i;
    if (i < passes && li < RL) {
      const int n = g + G * li;
      const float sc = ms.rsc[n];
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = hold[i][e] * sc * w[e];
      put(n, v);
    }
  }
  for (int i = kClHold; i < passes; ++i) {
    const int li = t / CH + RP * i;
    if (li >= RL) break;
    const int n = g + G * li;
    float v[8];
    in_load8(p, ms, in, n, col, v);
    const float sc = ms.rsc[n];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] *= sc * w[e];
    put(n, v);
  }
  if (!split) {
    cl_op_ready(p, ms, st);
    // the rows' 1/RMS from both halves, while the MMAs run: each CTA stores
    // its half's sums of squares into its partner's ms.ssp (counted on the
    // partner's ms.psx); the drain's barrier publishes ms.inv
    if (t < R) {
      const uint32_t pr = uint32_t(st.r ^ 1);
      cl_st1_async(cl_map(smem_u32(&ms.ssp[t]), pr), ms.ssx[t], cl_map(smem_u32(&ms.psx), pr));
    }
  } else {
    cev(p, st, CEV_OPREADY);
  }
  // both halves' statistics of every row: the other half's R sums of
  // squares, split also the sum of squares and scale of the own half's rows
  // that the three other CTAs built
  int* f = &ms.flag[st.fseq++ & 1];
  if (t == 0) {
    mbar_expect_tx(&ms.psx, uint32_t(R) * 4u + (split ? uint32_t(R - RL) * 8u : 0u));
    *f = cl_mwait(p, &ms.psx, st.pseq & 1);
  }
  ++st.pseq;
  named_bar(CBAR_CONS, kClCons);
  if (!*f) return false;
  cev(p, st, CEV_SSYNC);
  if (t < R) ms.inv[t] = rsqrtf((ms.ssx[t] + ms.ssp[t]) / float(p.d) + p.eps) / ms.rsc[t];
  return true;
}

// Frames b = r (mod 8) run attention in CTA r: activation row n (frame n /
// P, position n % P) lands in CTA (n / P) % 8 as its local row
// ((n / P) / 8) P + n % P.
__device__ __forceinline__ int att_dst(int n, int P) { return (n / P) % kCl; }
__device__ __forceinline__ int att_local(int n, int P) { return ((n / P) / kCl) * P + n % P; }
__device__ __forceinline__ int att_rows(int B, int P, int r) { return r < B ? ((B - 1 - r) / kCl + 1) * P : 0; }

// Drain the accumulator (128 weight rows x R activation rows, scaled by
// ms.inv per row) straight into the consumers' receive buffers with
// asynchronous stores counted on their ms.prx.  PUSH_ATT: row n of tile tq,
// K half h goes to the frame's attention CTA as recv[local row][tq][h][128];
// PUSH_GU: rows m of gate/up tile tq go to the CTA that applies SwiGLU to
// them, 4 (tq % 2) + m / 32, as recv[n][tq / 2][h][m % 32]; PUSH_HEAD: rows m
// of the tile go to the member of the CTA pair that completes them (m < 64:
// the K-half-0 CTA) as recv[n][h][m % 64].  Each warp moves 32 features x 8
// rows at a time (warps w and w + 4 share a lane quarter and take alternate
// 8-row chunks) through 1 KB of its own (the operand region is free once
// the MMAs are done), 8 consecutive features per lane.
enum { PUSH_ATT = 0, PUSH_GU = 1, PUSH_HEAD = 2 };
template <int MODE>
__device__ bool cl_drain_push(const CParams& p, CMisc& ms, CState& st, uint8_t* smem, int R, int P) {
  if (!cl_wait_acc(p, ms, st)) return false;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q = warp & 3, ch = warp >> 2;
  const int tq = st.r >> 1, h = st.r & 1;
  float* tp = reinterpret_cast<float*>(smem + kClOffOp) + warp * 256;   // [8 rows][32 features]
  const uint32_t recv = smem_u32(smem + kClOffRecv), bar = smem_u32(&ms.prx);
  const int f = lane >> 2, k8 = (lane & 3) * 8;   // this lane's row in the chunk and its features
  for (int col = ch * 8; col < R; col += 16) {   // warp-uniform; the two warps of a lane quarter alternate
    float v[8];
    tmem_ld8(ms.tmem_base + (uint32_t(q * 32) << 16) + uint32_t(col), v);
#pragma unroll
    for (int i = 0; i < 8; ++i) tp[i * 32 + lane] = v[i];
    __syncwarp();
    const int n = col + f;
    if (n < R) {
      const float sc = ms.inv[n];
      const float4 a = *reinterpret_cast<const float4*>(tp + f * 32 + k8);
      const float4 b = *reinterpret_cast<const float4*>(tp + f * 32 + k8 + 4);
      int dst;
      uint32_t off;   // byte offset in the destination's receive buffer
      if (MODE == PUSH_ATT) {
        dst = att_dst(n, P);
        off = uint32_t(((att_local(n, P) * 4 + tq) * 2 + h) * kTileM + q * 32 + k8) * 4;
      } else if (MODE == PUSH_GU) {
        dst = 4 * (tq & 1) + q;
        off = uint32_t(((n * 2 + (tq >> 1)) * 2 + h) * 32 + k8) * 4;
      } else {
        dst = (st.r & ~1) | (q >> 1);
        off = uint32_t((n * 2 + h) * 64 + (q & 1) * 32 + k8) * 4;
      }
      const uint32_t da = cl_map(recv + off, uint32_t(dst)), db = cl_map(bar, uint32_t(dst));
      cl_st4_async(da, make_float4(a.x * sc, a.y * sc, a.z * sc, a.w * sc), db);
      cl_st4_async(da + 16, make_float4(b.x * sc, b.y * sc, b.z * sc, b.w * sc), db);
    }
    __syncwarp();
  }
  tc_fence_before();
  return true;
}
// Wait (all consumer threads) until this CTA's share of the pushed partial
// products has landed: `bytes` of them (set here, before or after the peers'
// stores: a phase needs this arrival as well as the bytes).
__device__ bool cl_wait_recv(const CParams& p, CMisc& ms, CState& st, uint32_t bytes) {
  if (bytes == 0) return true;
  int* f = &ms.flag[st.fseq++ & 1];
  if (threadIdx.x == 0) {
    mbar_expect_tx(&ms.prx, bytes);
    *f = cl_mwait(p, &ms.prx, st.rseq & 1);
  }
  ++st.rseq;
  named_bar(CBAR_CONS, kClCons);
  return *f != 0;
}

// Drain the accumulator of an O or down tile (rows m0 .. m0+127 of the
// residual stream) into the residual rows n < R.  Each warp drains 32
// features x 8 rows at a time (alternate chunks with the other warp of its
// lane quarter), transposes them through 1 KB of shared
// memory (the start of the operand region, whose normalised operand the
// tensor cores read before any peer could reach the next one) and adds 4 consecutive features per thread
// with one vector reduction.  emb: also add the frame's code embedding
// (step k >= 2, layer 0, first kv group).
__device__ bool cl_drain_resid(const CParams& p, CMisc& ms, CState& st, uint8_t* smem, float* xrows, int R, int m0,
                               const uint16_t* emb) {
  if (!cl_wait_acc(p, ms, st)) return false;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q = warp & 3, ch = warp >> 2;
  float* tp = reinterpret_cast<float*>(smem + kClOffOp) + warp * 256;   // [8 rows][32 features]
  const int mq = m0 + q * 32;
  for (int col = ch * 8; col < R; col += 16) {   // warp-uniform; the two warps of a lane quarter alternate
    float v[8];
    tmem_ld8(ms.tmem_base + (uint32_t(q * 32) << 16) + uint32_t(col), v);
#pragma unroll
    for (int i = 0; i < 8; ++i) tp[i * 32 + lane] = v[i];
    __syncwarp();
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
      const int f = pass * 4 + (lane >> 3), k4 = (lane & 7) * 4, n = col + f;
      if (n < R) {
        float4 a = *reinterpret_cast<const float4*>(tp + f * 32 + k4);
        if (emb) {
          const uint2 e = *reinterpret_cast<const uint2*>(emb + size_t(ms.code[n]) * p.d + mq + k4);
          a.x += e16_to_f32(e.x, p.embed_f16); a.y += e16_to_f32(e.x >> 16, p.embed_f16);
          a.z += e16_to_f32(e.y, p.embed_f16); a.w += e16_to_f32(e.y >> 16, p.embed_f16);
        }
        red_add_v4_f32(xrows + size_t(n) * p.d + mq + k4, a);
      }
    }
    __syncwarp();
  }
  tc_fence_before();
  return true;
}

// ------------------------------------------------------------ the tasks
__device__ __forceinline__ float* cl_x(const CParams& p, int k) { return p.x + size_t(k - 1) * 2 * p.B * p.d; }

// The code each frame's step-k input embeds (k >= 2): the previous step's
// decision, or the forced one; out of range latches QP_ERR_BAD_TOKEN and is
// clamped.  Waits for the previous step's decisions first.
__device__ bool cl_step_codes(const CParams& p, CMisc& ms, CState& st, int k) {
  if (!cl_wait_ctr(p, ms, st, p.head_done + (k - 2), unsigned(p.n_head * kCl))) return false;
  const int t = threadIdx.x;
  if (t < p.B) {
    int code = unpack_argmax_index(__ldcg(p.best + size_t(k - 2) * p.B + t));
    if (p.forced) code = p.forced[size_t(t) * p.n_steps + (k - 2)];
    if (code < 0 || code >= p.V) {
      set_status(p.status, QP_ERR_BAD_TOKEN);
      code = code < 0 ? 0 : p.V - 1;
    }
    ms.code[t] = code;
  }
  named_bar(CBAR_CONS, kClCons);
  return true;
}

// Projection unit u of step k's inputs (tile u / (th/128), K slice u %
// (th/128)).  Step 1: rows 2b = H_b and 2b+1 = E0[q0_b], the first two
// positions of frame b (H and q0 feed the residual loop: "拆解 Qwen3-TTS：
// OpenVINO 移植过程中的图分离与调度实践", section 1; their order is a reading).
// Step k >= 2 with Talker-wide code tables: row b = E[k-2][the frame's
// code].  Each row's slice is scaled by 2^-e into f16's range (e from the
// slice's mean square) and the partial product by 2^e; the K slice 0 unit
// adds the bias.
template <bool EXT>
__device__ bool cl_proj(const CParams& p, CMisc& ms, CState& st, uint8_t* smem, const Task& tk) {
  const int k = EXT ? tk.k : 1;
  if (k > 1 && !cl_step_codes(p, ms, st, k)) return false;
  const int t = threadIdx.x, R = k == 1 ? 2 * p.B : p.B, np = cl_npad(R), n8 = np / 8;
  const int nks = p.th / kKs, mt = tk.job / nks, ks = tk.job % nks;
  uint16_t* op = reinterpret_cast<uint16_t*>(smem + kClOffOp);
  const int c = t & 15, kl = c * 8;
  for (int n = t >> 4; n < np; n += kClCons / 16) {   // warp-uniform: np is a multiple of 16
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (n < R) {
      if (k > 1) {
        ld8e(p.embed[k - 2] + size_t(ms.code[n]) * p.th + ks * kKs + kl, p.embed_f16, v);
      } else if ((n & 1) == 0) {
        const float* hr = p.H + size_t(n >> 1) * p.th + ks * kKs + kl;
        const float4 a = __ldg(reinterpret_cast<const float4*>(hr));
        const float4 e = __ldg(reinterpret_cast<const float4*>(hr + 4));
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = e.x; v[5] = e.y; v[6] = e.z; v[7] = e.w;
      } else {
        int q = p.q0[n >> 1];
        if (q < 0 || q >= p.q0_vocab) {
          if (c == 0 && mt == 0 && ks == 0) set_status(p.status, QP_ERR_BAD_TOKEN);
          q = q < 0 ? 0 : p.q0_vocab - 1;
        }
        ld8e(p.e0 + size_t(q) * p.th + ks * kKs + kl, p.embed_f16, v);
      }
    }
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) ss += v[e] * v[e];
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const int ex = range_exp(ss / float(kKs));
    const float sc = exp2i(-ex);
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] *= sc;
    if (n < R) {
      *reinterpret_cast<uint4*>(op + op_idx(n, kl, n8)) = pack8h(v);
      if (c == 0) ms.inv[n] = exp2i(ex);
    }
  }
  cl_op_ready(p, ms, st);
  if (!cl_wait_acc(p, ms, st)) return false;
  // as the O and down drains: 32 features x 8 rows per warp through 1 KB of
  // shared memory (the operand's, read by the finished MMAs), 4 features per
  // reduction, each row scaled by its 2^e and the bias added by K slice 0
  const int warp = t >> 5, lane = t & 31, q = warp & 3, ch = warp >> 2, mq = mt * kTileM + q * 32;
  const int k4 = (lane & 7) * 4;
  const float4 bias = ks == 0 ? __ldg(reinterpret_cast<const float4*>(p.b_proj + mq + k4)) : make_float4(0.f, 0.f, 0.f, 0.f);
  float* tp = reinterpret_cast<float*>(smem + kClOffOp) + warp * 256;   // [8 rows][32 features]
  float* xk = cl_x(p, k);
  for (int col = ch * 8; col < R; col += 16) {   // warp-uniform; the two warps of a lane quarter alternate
    float v[8];
    tmem_ld8(ms.tmem_base + (uint32_t(q * 32) << 16) + uint32_t(col), v);
#pragma unroll
    for (int i = 0; i < 8; ++i) tp[i * 32 + lane] = v[i];
    __syncwarp();
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
      const int f = pass * 4 + (lane >> 3), n = col + f;
      if (n < R) {
        const float4 a = *reinterpret_cast<const float4*>(tp + f * 32 + k4);
        const float sc = ms.inv[n];
        red_add_v4_f32(xk + size_t(n) * p.d + mq + k4,
                       make_float4(a.x * sc + bias.x, a.y * sc + bias.y, a.z * sc + bias.z, a.w * sc + bias.w));
      }
    }
    __syncwarp();
  }
  tc_fence_before();
  cl_publish(p, st, p.proj_done + (k - 1));
  return true;
}


// The wait before a step's layer-l attention job and where its input rows
// come from.  Step k >= 2, layer 0: with code tables as wide as the hidden
// size the previous step's decisions (each frame's code, or the forced one)
// select the code embedding rows; with Talker-wide tables the step's
// projection units wrote the rows.
template <bool EXT>
__device__ bool cl_att_input(const CParams& p, CMisc& ms, CState& st, const Task& tk, InSrc& in) {
  const int k = tk.k, l = tk.l;
  in.x = cl_x(p, k); in.emb = nullptr; in.row_mul = 1; in.row_add = 0;
  if (l > 0) return cl_wait_ctr(p, ms, st, p.mlp_done + (k - 1) * p.L + (l - 1), unsigned(p.n_mlp * kCl));
  if (k == 1 || cl_proj_in<EXT>(p)) return cl_wait_ctr(p, ms, st, p.proj_done + (k - 1), unsigned(p.n_proj));
  if (!cl_step_codes(p, ms, st, k)) return false;
  in.x = nullptr;
  in.emb = p.embed[k - 2];
  return true;
}

// Attention job j of layer l at step k, through the O operand: the QKV
// GEMM over this CTA's tile and K half, then for the frames b = r (mod 8),
// one warp per (frame, q head), the frame's q|k|v from the peers' partials,
// per-head RMSNorm and RoPE of the new position(s), KV append (by the head-0
// warp, into this CTA's tensor memory), causal softmax over positions 0..pos and the head's output written
// into every peer's O operand.  Lane l holds dims 4l..4l+3 of every
// 128-vector; the scores of 16 positions are 16 partial dot products per
// lane, summed by one reduce-scatter.
template <bool SPLIT, bool EXT>
__device__ bool cl_qkv(const CParams& p, CMisc& ms, CState& st, uint8_t* smem, const Task& tk) {
  const int k = tk.k, l = tk.l, R = cl_rows(p, tk), np = cl_npad(R), n8 = np / 8;
  InSrc in;
  if (!cl_att_input<EXT>(p, ms, st, tk, in)) return false;
  if (!cl_build_norm<SPLIT>(p, ms, st, smem, in, p.layer[l].attn_norm, R)) return false;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, fq = warp & 3, hh = warp >> 2;
  const int P = k == 1 ? 2 : 1, pos0 = k == 1 ? 0 : k;
  // warp w: q head hh = w / 4 of frame b = r + 8 (w % 4), whose KV cache for
  // kv head j sits in lane quarter w % 4 of this CTA's tensor memory (the
  // cluster keeps kv head j at every layer and step)
  const int b = st.r + kCl * fq;
  const uint32_t kvt = ms.tmem_base + (uint32_t(fq * 32) << 16) + kClKvCol + uint32_t(l) * kClKvColsPerLayer;
  // the positions of earlier steps (written by the head-0 warp), read while the MMAs run
  uint32_t kc[2 * kMaxCtx], vc[2 * kMaxCtx];
  const bool cached = b < p.B && pos0 > 0;   // warp-uniform
  if (cached) {
    tc_fence_after();
    tmem_ld32(kvt, kc);
    tmem_ld32(kvt + 2 * kMaxCtx, vc);
  } else {
#pragma unroll
    for (int i = 0; i < 2 * kMaxCtx; ++i) kc[i] = vc[i] = 0u;
  }
  // the head norms' weights and the new positions' RoPE factors, also while the MMAs run
  const CLayer& L = p.layer[l];
  const float4 qnw = __ldg(reinterpret_cast<const float4*>(L.q_norm + lane * 4));
  const float4 knw = __ldg(reinterpret_cast<const float4*>(L.k_norm + lane * 4));
  float2 cs[4];   // position pos0's (step 1 reloads them for position 1)
#pragma unroll
  for (int e = 0; e < 4; ++e) cs[e] = __ldg(p.rope_cs + pos0 * 64 + ((lane * 4 + e) & 63));
  // this CTA's O operand will hold R rows x 256 columns of f16, written by
  // the peers' attention warps
  if (threadIdx.x == 0 && st.r < p.d / kTileM) mbar_expect_tx(&ms.opx, uint32_t(R) * 512u);
  if (!cl_drain_push<PUSH_ATT>(p, ms, st, smem, R, P)) return false;
  // this CTA's frames' q|k|v: 4 tiles x 2 K halves x 128 per row
  if (!cl_wait_recv(p, ms, st, uint32_t(att_rows(p.B, P, st.r)) * 4096u)) return false;
  cev(p, st, CEV_S1);
  if (cached) tmem_wait_ld2(kc, vc);
  const float scale = rsqrtf(float(kHeadDim));
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  const float* recv = reinterpret_cast<const float*>(smem + kClOffRecv) + lane * 4;
  const uint32_t opsz = uint32_t(np) * kKs * 2;
  const uint32_t o0 = smem_u32(smem + kClOffOp2) + uint32_t(hh) * opsz;
  const int n_dst = min(kCl, p.d / kTileM);   // the CTAs with an O tile
  if (b < p.B) {
    float4 kprev = z4, vprev = z4;   // step 1: position 0's k and v, for position 1
    for (int pp = 0; pp < P; ++pp) {
      const int n = b * P + pp, pos = pos0 + pp;
      // the frame's q (head hh), k and v: the two K halves of tiles hh, 2 and 3
      float4 v4[3];
      const int nl = att_local(n, P);
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        const int tq = i == 0 ? hh : i + 1;
        const float* a = recv + ((nl * 4 + tq) * 2) * kTileM;
        const float4 h0 = *reinterpret_cast<const float4*>(a), h1 = *reinterpret_cast<const float4*>(a + kTileM);
        v4[i] = make_float4(h0.x + h1.x, h0.y + h1.y, h0.z + h1.z, h0.w + h1.w);
      }
      if (lane == 0 && threadIdx.x == 0) cl_ev(p, st.evi, 0, CEV_SUB, st.task);
      if (pp > 0)
#pragma unroll
        for (int e = 0; e < 4; ++e) cs[e] = __ldg(p.rope_cs + pos * 64 + ((lane * 4 + e) & 63));
      float4 knew, qn;
      norm_rope_w2(v4[1], knw, v4[0], qnw, cs, p.eps, lane, knew, qn);
      const float4 vnew = v4[2];
      if (hh == 0) {   // the new position into the cache
        tmem_st2(kvt + 2 * uint32_t(pos), pack4_f16(knew.x, knew.y, knew.z, knew.w));
        tmem_st2(kvt + 2 * kMaxCtx + 2 * uint32_t(pos), pack4_f16(vnew.x, vnew.y, vnew.z, vnew.w));
      }
      float part[16];   // positions after pos (masked below) skipped: pos is the same in every lane
#pragma unroll
      for (int tt = 0; tt < kMaxCtx; ++tt) {
        part[tt] = 0.f;
        if (tt <= pos) {
          const float4 kk = tt < pos0 ? unpack4_f16(make_uint2(kc[2 * tt], kc[2 * tt + 1])) : (tt == pos ? knew : kprev);
          part[tt] = qn.x * kk.x + qn.y * kk.y + qn.z * kk.z + qn.w * kk.w;
        }
      }
      if (lane == 0 && threadIdx.x == 0) cl_ev(p, st.evi, 0, CEV_SUB, st.task);
      const float rsum = reduce_scatter16(part, lane);   // lanes 2t and 2t + 1: position t
      const bool valid = ((lane >> 1) & 15) <= pos;
      const float sc = valid ? rsum * scale : -INFINITY;
      float mx = sc;
#pragma unroll
      for (int o = 16; o >= 2; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float e = valid ? expf(sc - mx) : 0.f;
      float den = e;
#pragma unroll
      for (int o = 16; o >= 2; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
      const float pr = den > 0.f ? e / den : 0.f;
      float4 o1 = z4;
#pragma unroll
      for (int tt = 0; tt < kMaxCtx; ++tt) {
        if (tt <= pos) {   // warp-uniform
          const float4 vv = tt < pos0 ? unpack4_f16(make_uint2(vc[2 * tt], vc[2 * tt + 1])) : (tt == pos ? vnew : vprev);
          const float w = __shfl_sync(0xffffffffu, pr, 2 * tt);
          o1.x += w * vv.x; o1.y += w * vv.y; o1.z += w * vv.z; o1.w += w * vv.w;
        }
      }
      if (lane == 0 && threadIdx.x == 0) cl_ev(p, st.evi, 0, CEV_SUB, st.task);
      // row n of the O operand (K = the group's 256 columns: head hh in slice hh) in every CTA
      const uint2 hv = pack4_f16(o1.x, o1.y, o1.z, o1.w);
      const uint32_t a = o0 + op_idx(n, lane * 4, n8) * 2;
      const uint32_t xbar = smem_u32(&ms.opx);
      for (int dst = 0; dst < n_dst; ++dst) cl_st2_async(cl_map(a, uint32_t(dst)), hv, cl_map(xbar, uint32_t(dst)));
      kprev = knew;
      vprev = vnew;
    }
    if (hh == 0) {   // the cache stores done before the barriers that order the next step's loads
      tmem_wait_st();
      tc_fence_before();
    }
  }
  cev(p, st, CEV_WORK);
  return true;   // each peer's MMA warp waits until its O operand's rows have landed
}

// O projection of attention job j (after cl_qkv): tile r of W_o over the
// group's 256 columns, added into the residual stream.
template <bool EXT>
__device__ bool cl_out(const CParams& p, CMisc& ms, CState& st, uint8_t* smem, const Task& tk) {
  const int R = cl_rows(p, tk);
  const bool mine = cl_nsl(p, tk) > 0;
  if (mine) {
    const uint16_t* emb =
        (tk.kind == T_O && tk.k > 1 && tk.l == 0 && tk.job == 0 && !cl_proj_in<EXT>(p)) ? p.embed[tk.k - 2] : nullptr;
    if (!cl_drain_resid(p, ms, st, smem, cl_x(p, tk.k), R, st.r * kTileM, emb)) return false;
  }
  unsigned* ctr = tk.kind == T_O ? p.att_done + (tk.k - 1) * p.L + tk.l : p.mlp_done + (tk.k - 1) * p.L + tk.l;
  if (tk.kind == T_O && p.withhold >= 0 && blockIdx.x == 0 && tk.k == 1 && tk.l == 0) {
    named_bar(CBAR_CONS, kClCons);   // a test of the failure path: this count goes missing
    return true;
  }
  cl_publish(p, st, ctr);
  return true;
}

// MLP job m of layer l at step k, through the down operand: gate/up over
// this CTA's tile and K half, then SwiGLU of columns 32r .. 32r+31 of the
// job's 256 from the peers' partials, written into every peer's down operand.
template <bool SPLIT>
__device__ bool cl_gu(const CParams& p, CMisc& ms, CState& st, uint8_t* smem, const Task& tk) {
  const int k = tk.k, l = tk.l, R = cl_rows(p, tk), np = cl_npad(R), n8 = np / 8;
  if (!cl_wait_ctr(p, ms, st, p.att_done + (k - 1) * p.L + l, unsigned(p.n_att * kCl))) return false;
  InSrc in{cl_x(p, k), nullptr, 1, 0};
  if (!cl_build_norm<SPLIT>(p, ms, st, smem, in, p.layer[l].ffn_norm, R)) return false;
  // this CTA's down operand will hold R rows x 256 columns of f16, written by the peers
  if (threadIdx.x == 0 && st.r < p.d / kTileM) mbar_expect_tx(&ms.opx, uint32_t(R) * 512u);
  if (!cl_drain_push<PUSH_GU>(p, ms, st, smem, R, 1)) return false;
  // this CTA's 32 columns of gate and up, both K halves: 512 B per row
  if (!cl_wait_recv(p, ms, st, uint32_t(R) * 512u)) return false;
  cev(p, st, CEV_S1);
  const int t = threadIdx.x, c4 = t & 7, r = st.r;
  const int tg = r >> 2, m = 32 * (r & 3) + 4 * c4;   // the gate (and up) tile of the columns, row in tile
  const uint32_t opsz = uint32_t(np) * kKs * 2;
  const float* recv = reinterpret_cast<const float*>(smem + kClOffRecv) + 4 * c4;   // [n][gate|up][half][32]
  const uint32_t o0 = smem_u32(smem + kClOffOp2) + uint32_t(tg) * opsz;   // slice c / 128 = r / 4
  const int n_dst = min(kCl, p.d / kTileM);   // the CTAs with a down tile
  for (int n = t >> 3; n < R; n += kClCons / 8) {
    const float* a = recv + n * 128;
    const float4 g0 = *reinterpret_cast<const float4*>(a), g1 = *reinterpret_cast<const float4*>(a + 32);
    const float4 u0 = *reinterpret_cast<const float4*>(a + 64), u1 = *reinterpret_cast<const float4*>(a + 96);
    const uint2 hv = pack4_f16(silu_f(g0.x + g1.x) * (u0.x + u1.x), silu_f(g0.y + g1.y) * (u0.y + u1.y),
                               silu_f(g0.z + g1.z) * (u0.z + u1.z), silu_f(g0.w + g1.w) * (u0.w + u1.w));
    const uint32_t d = o0 + op_idx(n, m, n8) * 2, xbar = smem_u32(&ms.opx);
    for (int dst = 0; dst < n_dst; ++dst) cl_st2_async(cl_map(d, uint32_t(dst)), hv, cl_map(xbar, uint32_t(dst)));
  }
  cev(p, st, CEV_WORK);
  return true;   // each peer's MMA warp waits until its down operand's rows have landed
}

// Head job hj at step k: logits 512 hj .. 512 hj + 511 of the step's head
// for every frame's last position; CTA r completes rows 64 (r%2) .. +63 of
// tile r/2, writes them out if asked and folds their argmax (lowest index
// on ties) into the frame's decision word.
template <bool SPLIT>
__device__ bool cl_head(const CParams& p, CMisc& ms, CState& st, uint8_t* smem, const Task& tk) {
  const int k = tk.k, R = p.B;
  if (!cl_wait_ctr(p, ms, st, p.mlp_done + (k - 1) * p.L + (p.L - 1), unsigned(p.n_mlp * kCl))) return false;
  InSrc in{cl_x(p, k), nullptr, k == 1 ? 2 : 1, k == 1 ? 1 : 0};
  if (!cl_build_norm<SPLIT>(p, ms, st, smem, in, p.out_norm, R)) return false;
  if (!cl_drain_push<PUSH_HEAD>(p, ms, st, smem, R, 1)) return false;
  // this CTA's 64 logits rows of the tile, both K halves: 512 B per frame
  if (!cl_wait_recv(p, ms, st, uint32_t(R) * 512u)) return false;
  cev(p, st, CEV_S1);
  const int t = threadIdx.x, mg = t & 7, n = t >> 3, r = st.r;
  const int m = 64 * (r & 1) + 8 * mg;
  unsigned long long key = 0ull;
  if (n < R) {
    const float* part = reinterpret_cast<const float*>(smem + kClOffRecv) + n * 128 + 8 * mg;   // [n][half][64]
    const float4 a0 = *reinterpret_cast<const float4*>(part), a1 = *reinterpret_cast<const float4*>(part + 4);
    const float4 b0 = *reinterpret_cast<const float4*>(part + 64), b1 = *reinterpret_cast<const float4*>(part + 68);
    const float lg[8] = {a0.x + b0.x, a0.y + b0.y, a0.z + b0.z, a0.w + b0.w,
                         a1.x + b1.x, a1.y + b1.y, a1.z + b1.z, a1.w + b1.w};
    const int v0 = 512 * tk.job + kTileM * (r >> 1) + m;
    if (p.out_logits) {
      float* o = p.out_logits + (size_t(n) * p.n_steps + (k - 1)) * p.V + v0;
      *reinterpret_cast<float4*>(o) = make_float4(lg[0], lg[1], lg[2], lg[3]);
      *reinterpret_cast<float4*>(o + 4) = make_float4(lg[4], lg[5], lg[6], lg[7]);
    }
    key = pack_argmax(lg[0], v0);
#pragma unroll
    for (int i = 1; i < 8; ++i) {
      const unsigned long long kk = pack_argmax(lg[i], v0 + i);
      key = kk > key ? kk : key;
    }
  }
#pragma unroll
  for (int o = 4; o >= 1; o >>= 1) {   // the frame's 8 threads (all lanes take part)
    const unsigned long long w = __shfl_xor_sync(0xffffffffu, key, o);
    key = w > key ? w : key;
  }
  if (n < R && mg == 0) atomicMax(p.best + size_t(k - 1) * p.B + n, key);
  cl_publish(p, st, p.head_done + (k - 1));
  return true;
}

template <bool SPLIT, bool EXT>
__device__ void cl_consumer(const CParams& p, CMisc& ms, uint8_t* smem) {
  CState st{0u, 0u, 0u, 0u, int(cl_rank()), 0, 0u};
  const Prog g = cl_prog(p);
  const int nt = cl_n_tasks<EXT>(p, g);
  for (int i = 0; i < nt; ++i) {
    const Task tk = cl_task<EXT>(p, g, i);
    st.task = i;
    cev(p, st, CEV_START);
    bool ok = true;
    switch (tk.kind) {
      case T_PROJ: ok = cl_proj<EXT>(p, ms, st, smem, tk); break;
      case T_QKV: ok = cl_qkv<SPLIT, EXT>(p, ms, st, smem, tk); break;
      case T_GU: ok = cl_gu<SPLIT>(p, ms, st, smem, tk); break;
      case T_HEAD: ok = cl_head<SPLIT>(p, ms, st, smem, tk); break;
      default: ok = cl_out<EXT>(p, ms, st, smem, tk); break;   // T_O, T_DOWN
    }
    if (!ok) return;
  }
  // the codes of every step, once the last step's decisions are in
  if (blockIdx.x == 0) {
    if (!cl_wait_ctr(p, ms, st, p.head_done + (p.n_steps - 1), unsigned(p.n_head * kCl))) return;
    for (int i = threadIdx.x; i < p.B * p.n_steps; i += kClCons) {
      const int b = i / p.n_steps, k = i % p.n_steps;
      p.out_codes[i] = unpack_argmax_index(__ldcg(p.best + size_t(k) * p.B + b));
    }
  }
}

// SPLIT: the build that shares the loads of a K half among four CTAs is
// compiled in (batches of kClSplitRows frames and more); without it the
// kernel's code stays smaller, which shows at small batches (119.8 vs 125.0
// us per step at one frame, measured).
template <bool SPLIT, bool EXT>
__global__ void __launch_bounds__(kClThreads, 1) k_frames_cluster(const CParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  CMisc& ms = *reinterpret_cast<CMisc*>(smem + kClOffMisc);
  const int t = threadIdx.x, warp = t >> 5;
  if (t == 0) {
    for (int i = 0; i < kClNW; ++i) { mbar_init(&ms.wfull[i], 1); mbar_init(&ms.wempty[i], 1); }
    mbar_init(&ms.opfull, 1);
    mbar_init(&ms.accfull, 1);
    mbar_init(&ms.mmadone, 1);
    mbar_init(&ms.opx, 1);
    mbar_init(&ms.prx, 1);
    mbar_init(&ms.psx, 1);
    mbar_init(&ms.nx, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tmem_alloc(&ms.tmem_base, kClTmemCols);
  tc_fence_before();
  cl_barrier_all();   // every CTA's barriers are initialised before any peer arrives on them
  tc_fence_after();

  if (warp < kClConsWarps) {
    cl_consumer<SPLIT, EXT>(p, ms, smem);
  } else if (warp == kClProdWarp) {
    if ((t & 31) == 0) cl_producer<EXT>(p, ms, smem);
    __syncwarp();
  } else if (warp == kClMmaWarp) {
    if ((t & 31) == 0) cl_mma<SPLIT, EXT>(p, ms, smem);
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(ms.tmem_base, kClTmemCols);
  cl_barrier_all();   // no CTA leaves while a peer may still use its shared memory
}

// ------------------------------------------------------------------ host
size_t cl_al256(size_t b) { return (b + 255) & ~size_t(255); }

struct ClLayout {
  size_t x, proj_done, att_done, mlp_done, head_done, best, abort_flag, zeroed, kv, total;
};
ClLayout cl_layout(const qp_geometry& g, int B) {
  ClLayout Lo{};
  const size_t steps = size_t(g.n_steps), L = size_t(g.layers);
  size_t o = 0;
  Lo.x = o;          o += cl_al256(steps * 2 * B * g.hidden * 4);
  Lo.proj_done = o;  o += cl_al256(steps * 4);
  Lo.att_done = o;   o += cl_al256(steps * L * 4);
  Lo.mlp_done = o;   o += cl_al256(steps * L * 4);
  Lo.head_done = o;  o += cl_al256(steps * 4);
  Lo.best = o;       o += cl_al256(steps * B * 8);
  Lo.abort_flag = o; o += 256;
  Lo.zeroed = o;
  Lo.total = o;
  return Lo;
}

constexpr int kClMaxDevices = 64;
// Per device: the kernel's shared-memory limit is set (1) and the clusters
// that fit at once (> 0), or no cluster launch is possible (-1).
std::atomic<int> g_cl_clusters[kClMaxDevices];

size_t cl_smem_bytes() { return kClOffMisc + sizeof(CMisc) + 1024; }

int cl_clusters(int dev) {
  std::atomic<int> local(0);
  std::atomic<int>* slot = dev >= 0 && dev < kClMaxDevices ? &g_cl_clusters[dev] : &local;
  int n = slot->load(std::memory_order_acquire);
  if (n != 0) return n;
  const int smem = int(cl_smem_bytes());
  if (cudaFuncSetAttribute(k_frames_cluster<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
      cudaFuncSetAttribute(k_frames_cluster<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
      cudaFuncSetAttribute(k_frames_cluster<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
      cudaFuncSetAttribute(k_frames_cluster<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
    cudaGetLastError();
    n = -1;
  } else {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = kCl; at[0].val.clusterDim.y = 1; at[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(kCl); cfg.blockDim = dim3(kClThreads); cfg.dynamicSmemBytes = size_t(smem);
    cfg.attrs = at; cfg.numAttrs = 1;
    int m = 0;
    int m2 = 0;
    int m3 = 0, m4 = 0;
    if (cudaOccupancyMaxActiveClusters(&m, k_frames_cluster<false, false>, &cfg) != cudaSuccess || m < 1 ||
        cudaOccupancyMaxActiveClusters(&m2, k_frames_cluster<true, false>, &cfg) != cudaSuccess || m2 < 1 ||
        cudaOccupancyMaxActiveClusters(&m3, k_frames_cluster<false, true>, &cfg) != cudaSuccess || m3 < 1 ||
        cudaOccupancyMaxActiveClusters(&m4, k_frames_cluster<true, true>, &cfg) != cudaSuccess || m4 < 1) {
      cudaGetLastError();
      n = -1;
    } else {
      n = std::min(std::min(m, m2), std::min(m3, m4));
    }
  }
  slot->store(n, std::memory_order_release);
  return n;
}

}  // namespace

size_t cluster_scratch_bytes(const qp_geometry& g, int bmax) { return cl_layout(g, bmax).total; }

bool cluster_ext(const qp_handle* h) {
  return h->wfmt == WF_Q8_0 || h->hfmt == WF_Q8_0 || h->g.code_embed_dim != h->g.hidden;
}

bool cluster_geometry_ok(const qp_geometry& g) {
  // hidden 512 or 1024: a row half of 256 or 512 columns is 32 or 64 chunks of 8, so each warp of an
  // operand build holds chunks of one row and the consumers cover whole rows per pass
  return g.head_dim == kHeadDim && g.n_q_heads == 2 * g.n_kv_heads && (g.hidden == 512 || g.hidden == 1024) &&
         g.ffn % 256 == 0 && g.vocab % 512 == 0 &&
         (g.code_embed_dim == g.hidden || g.code_embed_dim == g.talker_hidden) && g.talker_hidden % kKs == 0 &&
         g.n_steps + 1 <= kMaxCtx && g.layers <= kClMaxLayers;
}

bool cluster_supported(const qp_handle* h, const RunArgs& a) {
  if (!h->carena || !cluster_geometry_ok(h->g)) return false;
  // Q8_0 matrices (layers and projection, or heads) through their f16 hi and lo images
  if (h->wfmt == WF_Q8_0 && !h->layer[0].qkv.w16[0]) return false;
  if (h->hfmt == WF_Q8_0 && !h->head[0].w16[0]) return false;
  if (a.B < 1 || a.B > h->cmax_batch || a.B > kClusterMaxFrames) return false;
  if (a.temperature > 0.f) return false;
  return cl_clusters(h->device) > 0;
}

qp_status run_frames_cluster(qp_handle* h, const RunArgs& a, cudaStream_t s) {
  if (!cluster_supported(h, a)) return QP_ERR_ARG;
  const qp_geometry& g = h->g;
  const int n_cl = std::min(cl_clusters(h->device), h->num_sms / kCl);
  if (n_cl < 1) return QP_ERR_ARG;
  const ClLayout Lo = cl_layout(g, a.B);
  uint8_t* base = static_cast<uint8_t*>(h->carena);
  CParams p{};
  p.d = g.hidden; p.qw = g.n_q_heads * kHeadDim; p.kvw = g.n_kv_heads * kHeadDim; p.F = g.ffn; p.V = g.vocab;
  p.th = g.talker_hidden; p.L = g.layers; p.n_kv = g.n_kv_heads; p.n_steps = g.n_steps; p.q0_vocab = g.q0_vocab;
  p.eps = g.rms_eps;
  p.embed_f16 = h->embed_f16;
  // 16-bit matrices as packed; Q8_0 matrices through their f16 hi and lo images
  auto hi = [](const PackedMat& m) {
    return reinterpret_cast<const uint16_t*>(m.fmt == WF_Q8_0 ? m.w16[0] : m.w);
  };
  auto lo = [](const PackedMat& m) {
    return m.fmt == WF_Q8_0 ? reinterpret_cast<const uint16_t*>(m.w16[1]) : nullptr;
  };
  p.w_proj = hi(h->proj); p.w_proj_lo = lo(h->proj); p.b_proj = h->b_proj; p.e0 = h->e0;
  p.proj_in = g.code_embed_dim != g.hidden;
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
  p.x = reinterpret_cast<float*>(base + Lo.x);
  p.proj_done = reinterpret_cast<unsigned*>(base + Lo.proj_done);
  p.att_done = reinterpret_cast<unsigned*>(base + Lo.att_done);
  p.mlp_done = reinterpret_cast<unsigned*>(base + Lo.mlp_done);
  p.head_done = reinterpret_cast<unsigned*>(base + Lo.head_done);
  p.best = reinterpret_cast<unsigned long long*>(base + Lo.best);
  p.abort_flag = reinterpret_cast<int*>(base + Lo.abort_flag);
  p.status = h->status;
  p.spin_limit = h->wait_ticks > 0 ? h->wait_ticks : kSpinLimit;
  p.withhold = h->withhold_gemm;
  p.trace = h->trace; p.trace_n = h->trace_phases;
  p.n_cl = n_cl;
  p.n_att = g.n_kv_heads; p.n_mlp = g.ffn / 256; p.n_head = g.vocab / 512;
  p.n_proj = (g.hidden / kTileM) * (g.talker_hidden / kKs);
  p.B = a.B; p.H = a.H; p.q0 = a.q0; p.out_codes = a.out_codes; p.out_logits = a.out_logits; p.forced = a.forced;

  if (cudaMemsetAsync(base, 0, Lo.zeroed, s) != cudaSuccess) {
    cudaGetLastError();
    return QP_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kCl; at[0].val.clusterDim.y = 1; at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeCooperative;
  at[1].val.cooperative = 1;
  cfg.gridDim = dim3(n_cl * kCl); cfg.blockDim = dim3(kClThreads); cfg.dynamicSmemBytes = cl_smem_bytes();
  // QP_CLUSTER_NO_COOP=1 drops the cooperative attribute (include/qp_debug.h): Nsight Compute
  // rejects a cooperative launch with a cluster dimension.  Correctness does not rest on it:
  // every wait is bounded and a cluster's CTAs are always scheduled together.
  static const bool no_coop = [] {
    const char* e = getenv("QP_CLUSTER_NO_COOP");
    return e && e[0] == '1';
  }();
  cfg.stream = s; cfg.attrs = at; cfg.numAttrs = no_coop ? 1 : 2;
  // the build that shares loads pays off once every step's rows reach kClSplitRows
  const bool split = a.B >= kClSplitRows, ext = cluster_ext(h);
  const cudaError_t e = ext ? (split ? cudaLaunchKernelEx(&cfg, k_frames_cluster<true, true>, p)
                                     : cudaLaunchKernelEx(&cfg, k_frames_cluster<false, true>, p))
                            : (split ? cudaLaunchKernelEx(&cfg, k_frames_cluster<true, false>, p)
                                     : cudaLaunchKernelEx(&cfg, k_frames_cluster<false, false>, p));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return QP_ERR_CUDA;
  }
  return QP_OK;
}

}  // namespace qp
