// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <stddef.h>

#include "../../include/qp.h"

namespace qp {

constexpr int kMaxLayers = 16;
constexpr int kMaxSteps = 15;
constexpr int kMaxCtx = kMaxSteps + 1;   // positions 0..n_steps
constexpr int kHeadDim = 128;
constexpr int kTileM = 128;              // weight rows per MMA tile
constexpr int kKs = 128;                 // K per slice
constexpr int kMaxNc = 128;              // frames (rows) per MMA N chunk
constexpr int kMaxVocab = 4096;

enum WFmt { WF_BF16 = 0, WF_Q8_0 = 1 };

// A weight matrix packed for the tensor cores: 128-row tiles, each the
// K-major core-matrix image [K/8][16][8 rows][8 k] of f16 (bf16 input,
// converted) or of int8 (Q8_0 input, with f16 scales [tile][K/128][4][128]).
// One 128-row x 128-K slice is contiguous: 32 KB (f16) or 16 KB + 1 KB.
struct PackedMat {
  uint8_t* w = nullptr;
  __half* scale = nullptr;
  int N = 0, K = 0;
  int fmt = 0;    // WF_BF16 (16-bit source, packed as f16) or WF_Q8_0
  // Q8_0 only: the weights d*q as two f16 images in the 16-bit packed layout,
  // hi = f16(d*q) and lo = f16(d*q - hi) (hi + lo = d*q exactly), for the
  // small-batch engine, which streams 16-bit slices and multiplies both.
  uint8_t* w16[2] = {nullptr, nullptr};
};

struct LayerW {
  PackedMat qkv;   // [q_width + 2*kv_width, hidden]: q rows, then k rows, then v rows
  PackedMat o;     // [hidden, q_width]
  PackedMat gu;    // [2*ffn, hidden]: gate rows, then up rows
  PackedMat down;  // [hidden, ffn]
  const float* attn_norm = nullptr;
  const float* q_norm = nullptr;
  const float* k_norm = nullptr;
  const float* ffn_norm = nullptr;
};

// Per-call arguments of the frame loop.
struct RunArgs {
  int B = 0;
  const float* H = nullptr;
  const int32_t* q0 = nullptr;
  int32_t* out_codes = nullptr;
  float* out_logits = nullptr;
  const int32_t* forced = nullptr;
  float temperature = 0.f;   // 0 => greedy
  int top_k = 0;
  const float* gumbel = nullptr;
};

// A state-slot call (include/qp_sched.h): mode 1 runs step 1 of new frames
// into their slots, mode 2 one step of rows at their own steps.  slots and
// steps are host arrays [B]; the rest are device pointers in caller order.
struct SlotArgs {
  int mode = 0;
  int B = 0;
  const int32_t* slots = nullptr;
  const int32_t* steps = nullptr;      // mode 2
  const float* H = nullptr;            // mode 1
  const int32_t* q0 = nullptr;         // mode 1
  const int32_t* codes_in = nullptr;   // mode 2
  int32_t* out_codes = nullptr;
  float* out_logits = nullptr;
  float temperature = 0.f;             // 0 => greedy; else Gumbel top-k with the caller's noise
  int top_k = 0;
  const float* gumbel = nullptr;       // device [B][vocab]: each row's noise for its one step, caller order
};

// Rows of the MMA operand buffer for R activation rows (chunks of <= 128).
inline size_t operand_rows(size_t R) {
  const size_t r16 = (R + 15) / 16 * 16;
  return r16 <= size_t(kMaxNc) ? r16 : (R + kMaxNc - 1) / kMaxNc * kMaxNc;
}

// Byte offsets of the kernel's scratch for batches of up to `bmax` frames.
struct Scratch {
  size_t x1, xk;                         // residual streams: step 1 [2B, d], later steps [B, d]
  size_t a1[5], ak[4], ahead;            // f16 operands: step 1 proj/qkv/o/gu/down, later qkv/o/gu/down, head
  size_t acc1_qkv, acck_qkv, acc1_gu, acck_gu, logits;
  size_t acc_qkv_b;                      // a second [2B, q|k|v] accumulator (small-batch engine)
  size_t kv;                             // [layer][frame][pos][k|v][kv_width] f16
  size_t sync;                           // start of the zeroed-per-call region
  size_t total;                          // sync + the largest sync region (B = bmax)
};
Scratch scratch_layout(const qp_geometry& g, int bmax);
// Bytes of the synchronisation region a call with B frames uses (zeroed at
// the start of every call): counters, sums of squares, argmax words,
// decisions, abort flag.
size_t sync_bytes(const qp_geometry& g, int B);

// Largest batch the small-batch engine serves (2B <= 128 activation rows at
// step 1: one tensor-core N chunk), and the largest it is chosen for
// automatically: its operand slices are built from f32 sources by every CTA
// that uses them, which beyond ~40 frames costs more per step on GB300 than
// the tile engine's shared finishing passes (measured: 205.5 vs 207.7 us per
// step at 40 frames, 221.7 vs 209.1 at 48).
constexpr int kSmallMaxFrames = 64;
constexpr int kSmallAutoFrames = 40;
// Largest batch the cluster engine serves (2B <= 64 activation rows at step
// 1: its operand and partial buffers share 64 KB of shared memory).  Where it
// serves a call, QP_ENGINE_AUTO takes it: measured on GB300 at the 1.7B
// geometry, 90.0 vs 136.0 us per step at 1 frame (small-batch engine),
// 99.2 vs 143.6 at 8, 135.6 vs 193.2 at 32.
constexpr int kClusterMaxFrames = 32;
// With Q8_0 matrices or Talker-wide code tables (the exporter's layout) the
// cluster engine is the faster one at every batch it serves (measured, against
// the small-batch engine: 133.7 vs 158.2 us per step at 1 frame, 179.3 vs 211.2
// at 32).
constexpr int kClusterExtAutoFrames = 1;

}  // namespace qp

struct qp_handle {
  qp_geometry g;
  int max_batch = 0;
  int device = 0;
  int num_sms = 0;
  bool loaded = false;
  int wfmt = qp::WF_BF16;       // projection and layer matrices
  int hfmt = qp::WF_BF16;       // lm-heads
  bool embed_f16 = false;       // the embedding tables (q0 and code tables) are f16, else bf16

  // weights (library-owned arena)
  void* warena = nullptr;
  size_t warena_bytes = 0;
  qp::PackedMat proj;
  const float* b_proj = nullptr;
  const uint16_t* e0 = nullptr;                 // [q0_vocab, talker_hidden] 16-bit (embed_f16)
  qp::LayerW layer[qp::kMaxLayers];
  const float* out_norm = nullptr;
  const uint16_t* embed[qp::kMaxSteps] = {};    // [vocab, code_embed_dim] 16-bit (embed_f16)
  const float* embed_ss[qp::kMaxSteps] = {};    // [vocab]: sum of squares of each row
  qp::PackedMat head[qp::kMaxSteps];            // [vocab, hidden]

  // scratch: persistent buffers then the per-call sync region
  void* sarena = nullptr;
  size_t sarena_bytes = 0;
  qp::Scratch scr;
  // the cluster engine's scratch (qp_cluster.cu), for batches of up to cmax_batch frames; null where
  // the geometry is not one it serves
  void* carena = nullptr;
  int cmax_batch = 0;
  // small fixed buffers
  void* farena = nullptr;
  int* status = nullptr;                        // device status word
  float2* rope_cs = nullptr;                    // [ctx][64] (cos, sin)
  float* H_stage = nullptr;                     // host-buffer entry point staging
  int32_t* q0_stage = nullptr;
  int32_t* codes_stage = nullptr;
  unsigned long long* trace = nullptr;          // optional phase trace (qp_debug.h)
  int trace_phases = 0;

  int engine = 0;                               // qp_engine (qp_debug.h)
  long long wait_ticks = 0;                     // spin limit of the kernels' waits (0: the default)
  int withhold_gemm = -1;                       // testing: one CTA skips its count of this GEMM
  bool deterministic = false;                   // qp_set_deterministic (tile engine, fixed-order sums)
  int clock_khz = 0;                            // the device's SM clock (kHz), for wait_ticks
};

namespace qp {
// persistent engine (qp_persistent.cu)
qp_status run_frames_persistent(qp_handle* h, const RunArgs& a, cudaStream_t s);
qp_status run_frames_static(qp_handle* h, const RunArgs& a, cudaStream_t s);
size_t persistent_smem_bytes();
// the Q8_0 build of the tile engine's kernel (qp_persistent_q8.cu)
qp_status run_tile_q8(qp_handle* h, const RunArgs& a, uint8_t* scratch, const Scratch& L, int bmax, cudaStream_t s);
// cluster engine (qp_cluster.cu): greedy frame loop, at most kClusterMaxFrames
size_t cluster_scratch_bytes(const qp_geometry& g, int bmax);
// Q8_0 matrices or Talker-wide code tables: the engine's extended instantiation
bool cluster_ext(const qp_handle* h);
bool cluster_geometry_ok(const qp_geometry& g);
bool cluster_supported(const qp_handle* h, const RunArgs& a);
qp_status run_frames_cluster(qp_handle* h, const RunArgs& a, cudaStream_t s);
// small-batch engine (qp_small.cu): 16-bit slices (Q8_0 matrices through
// their hi and lo images), at most kSmallMaxFrames
bool small_supported(const qp_handle* h, const RunArgs& a);
qp_status run_frames_small(qp_handle* h, const RunArgs& a, uint8_t* scratch, const Scratch& L, int bmax,
                           cudaStream_t s);
// the same with Gumbel top-k sampling, on the kernel built from qp_small_sampled.cu
qp_status run_frames_small_sampled(qp_handle* h, const RunArgs& a, uint8_t* scratch, const Scratch& L, int bmax,
                                   cudaStream_t s);
size_t small_smem_bytes();
// state-slot calls on the small-batch engine's kernel built from qp_small_slots.cu
qp_status run_slots_small(qp_handle* h, const SlotArgs& a, uint8_t* scratch, const Scratch& L, int bmax,
                          cudaStream_t s);
// the same with Gumbel top-k sampling, on the kernel built from qp_small_slots_sampled.cu
qp_status run_slots_small_sampled(qp_handle* h, const SlotArgs& a, uint8_t* scratch, const Scratch& L, int bmax,
                                  cudaStream_t s);
// load-time weight preparation (qp_weights.cu)
size_t packed_bytes(int fmt, int N, int K);
// Pack `rows` rows of a caller matrix [rows, K] (16-bit -- f16 if src_f16,
// else bf16 -- or a Q8_0 block stream) into rows [row0, row0 + rows) of the
// packed matrix dst (and, for Q8_0, of its f16 hi and lo images).
cudaError_t pack_rows(const void* src, int fmt, bool src_f16, int rows, int K, const PackedMat& dst, int row0,
                      cudaStream_t s);
// out[b][j] = tables[j][codes[b][j]] as f32 for b < B, j < n_tables
// (tables: a host array of n_tables <= kMaxSteps device pointers to [V, d]
// tables, f16 if f16, else bf16).
cudaError_t code_embeddings(const uint16_t* const* tables, int n_tables, int V, int d, const int32_t* codes, int B,
                            float* out, int* status, bool f16, cudaStream_t s);
// out[r] = sum_i E[r, i]^2 (f32) for a [rows, cols] 16-bit table (f16 if f16, else bf16).
cudaError_t row_sumsq_e16(const uint16_t* E, int rows, int cols, bool f16, float* out, cudaStream_t s);
}  // namespace qp
