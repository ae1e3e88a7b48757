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

enum WFmt { WF_BF16 = 0, WF_Q8_0 = 1 };

// A weight matrix [N, K] (HF [out, in]) in the library's own layout.
//   WF_BF16: w = bf16 bits, row-major [N, K]
//   WF_Q8_0: w = int8 values row-major [N, K]; scale = f16 [N, K/32]
struct QMat {
  const void* w = nullptr;
  const __half* scale = nullptr;
  int N = 0, K = 0;
  int fmt = WF_BF16;
};

// A weight matrix packed for the tensor cores: 128-row tiles, each the
// K-major core-matrix image [K/8][16][8 rows][8 k] of f16 (WF_BF16 input)
// or int8 (WF_Q8_0 input, with f16 scales [tile][K/128][4][128]).
struct PackedMat {
  uint8_t* w = nullptr;
  __half* scale = nullptr;
};

struct PackedLayer {
  PackedMat qkv, o, gu, down;
};

struct LayerW {
  QMat qkv;   // [q_width + 2*kv_width, hidden]: q rows, then k rows, then v rows
  QMat o;     // [hidden, q_width]
  QMat gu;    // [2*ffn, hidden]: gate rows, then up rows
  QMat down;  // [hidden, ffn]
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

}  // namespace qp

struct qp_handle {
  qp_geometry g;
  int max_batch = 0;
  int device = 0;
  int num_sms = 0;
  bool loaded = false;
  int wfmt = qp::WF_BF16;

  // weights (library-owned arena)
  void* warena = nullptr;
  size_t warena_bytes = 0;
  qp::QMat proj;
  const float* b_proj = nullptr;
  const uint16_t* e0 = nullptr;            // [q0_vocab, talker_hidden] bf16
  qp::LayerW layer[qp::kMaxLayers];
  const float* out_norm = nullptr;
  const uint16_t* embed[qp::kMaxSteps] = {};  // [vocab, hidden] bf16
  qp::QMat head[qp::kMaxSteps];            // [vocab, hidden]
  // the same matrices packed for the persistent tensor-core engine
  qp::PackedMat pproj;
  qp::PackedLayer player[qp::kMaxLayers];
  qp::PackedMat phead[qp::kMaxSteps];

  // scratch (sized for max_batch)
  void* sarena = nullptr;
  size_t sarena_bytes = 0;
  float* X = nullptr;          // [2*max_batch, hidden] residual stream
  uint16_t* act = nullptr;     // [2*max_batch, act_width] f16 GEMM operand
  int act_width = 0;
  float* qkv = nullptr;        // [2*max_batch, q_width + 2*kv_width]
  float* gu = nullptr;         // [2*max_batch, 2*ffn]
  float* kv = nullptr;         // [layers][max_batch][ctx][2][n_kv][128]
  float* logits = nullptr;     // [max_batch, vocab]
  int* status = nullptr;       // device status word
  uint16_t* pact = nullptr;    // f16 MMA operand, [chunk][K/8][Nc/8][8][8]
  unsigned int* sync_words = nullptr;  // grid-barrier counter, abort flag
  float2* rope_cs = nullptr;   // [ctx][64] (cos, sin)
  // staging for the host-buffer entry point
  float* H_stage = nullptr;
  int32_t* q0_stage = nullptr;
  int32_t* codes_stage = nullptr;
};

namespace qp {
// engine entry (qp_engine.cu): enqueue the whole frame loop on s
qp_status run_frames(qp_handle* h, const RunArgs& a, cudaStream_t s);
// persistent engine (qp_persistent.cu)
qp_status run_frames_persistent(qp_handle* h, const RunArgs& a, cudaStream_t s);
size_t packed_bytes(int fmt, int N, int K);
cudaError_t pack_matrix(const QMat& src, PackedMat& dst, cudaStream_t s);
size_t persistent_smem_bytes();
// the same kernel with its scratch in a static device array (qp_persistent.cu)
qp_status run_frames_static(qp_handle* h, const RunArgs& a, cudaStream_t s);
int launches_per_call(const qp_handle* h, int B, bool sampling);
// weight repack helpers (qp_engine.cu)
cudaError_t repack_q8_0(const uint8_t* blocks, int N, int K, int8_t* qs, __half* d, cudaStream_t s);
}  // namespace qp
