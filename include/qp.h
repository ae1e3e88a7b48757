/*
 * qp.h -- C ABI of the GB300 Code Predictor library (libqp.so).
 *
 * The library runs the per-frame Code Predictor loop of Qwen3-TTS: for every
 * audio frame, given the Talker's hidden state H and first-codebook token q0,
 * a 5-layer causal transformer takes 15 autoregressive steps and emits the
 * residual-codebook tokens q1..q15 (16 codebooks with q0).  Frames from many
 * requests are batched into one call.
 *
 *   - 15 fixed steps per frame, a preallocated KV cache, the whole frame loop
 *     run as one fixed GPU program instead of a host-driven sequence:
 *     "テキスト音声合成モデルを50ミリ秒未満で応答させる方法", section
 *     "Qwen3-TTSの最適化方法", item 3.
 *   - The predictor is a stateless batched step whose inputs are the frame's
 *     H (and q0) and whose outputs are the residual codes:
 *     "拆解 Qwen3-TTS：OpenVINO 移植过程中的图分离与调度实践", sections 1, 2.2.
 *   - Geometry, tensor names and shapes, Q8_0 storage, and the rule that a
 *     loader fails on missing or unmapped tensors: "rightkit-qts 0.2.3 -
 *     Qwen3-TTS 1.7B -> QTS GGUF", sections "Loader contract", "Expected
 *     verification shapes", "Upstream differences & verification scope".
 *   - Sampling stays caller-controlled (same page, "Usage"): the caller
 *     passes temperature, top-k and the Gumbel noise itself.
 *
 * Conventions for every entry point:
 *   - Device pointers are CUDA device addresses on the handle's device,
 *     owned by the caller, read/written asynchronously on the given stream.
 *   - qp_stream is a cudaStream_t passed as void*; NULL means the legacy
 *     default stream.
 *   - A call that returns anything but QP_OK enqueued nothing.
 *   - Errors the GPU detects (an out-of-range token, a wait on another
 *     CTA's work that ran out of time) are latched in a device status word;
 *     qp_get_device_status reads and clears it.  Kernels never trap: a bad token is clamped for addressing
 *     and reported.
 *   - A handle may be used from one host thread at a time, and its calls
 *     share one scratch area (activations, KV cache, synchronisation
 *     words): calls on one handle must not overlap on the GPU, so a caller
 *     that uses several streams orders them (events) or uses one handle per
 *     stream.  The KV state slots of include/qp_sched.h live in that same
 *     area, so a prediction call on a handle ends the frames in its slots.
 */
#ifndef QP_H
#define QP_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QP_ABI_VERSION 1

typedef enum qp_status {
  QP_OK = 0,
  QP_ERR_ARG = 1,            /* null pointer, B out of range, bad geometry  */
  QP_ERR_STATE = 2,          /* weights not loaded / already loaded          */
  QP_ERR_WEIGHT_MISSING = 3, /* a required tensor was not supplied           */
  QP_ERR_WEIGHT_SHAPE = 4,   /* shape differs from the geometry              */
  QP_ERR_WEIGHT_DTYPE = 5,   /* storage type not accepted for that tensor    */
  QP_ERR_CUDA = 6,           /* a CUDA runtime call failed                   */
  QP_ERR_TIMEOUT = 7,        /* device: a wait on another CTA's work ran out */
  QP_ERR_BAD_TOKEN = 8,      /* device: q0 or a forced code out of range     */
  QP_ERR_OOM = 9,            /* device allocation failed in create/load      */
  QP_ERR_UNKNOWN_WEIGHT = 10,/* a supplied name is not a predictor tensor    */
  QP_ERR_DUPLICATE_WEIGHT = 11
} qp_status;

/* Storage types of weight tensors. */
typedef enum qp_dtype {
  QP_BF16 = 0,
  QP_F16 = 1,
  QP_F32 = 2,
  QP_Q8_0 = 3   /* blocks of 32 along the input dim: {f16 d; int8 q[32]},
                   34 bytes, value = d * q (GGUF Q8_0)                        */
} qp_dtype;

/* Predictor geometry.  qp_default_geometry fills the 1.7B Code Predictor:
 * hidden 1024, 5 layers, 16 q-heads / 8 kv-heads of 128, FFN 3072, 2048-entry
 * codebooks, 15 steps, Talker width 2048, 1024-wide code embeddings that
 * enter unprojected, 2048-entry q0 table, RMSNorm eps 1e-6, RoPE theta 1e6.
 * Supported: head_dim 128; n_q_heads a multiple of n_kv_heads;
 * code_embed_dim == hidden (code embeddings enter the stream unprojected) or
 * code_embed_dim == talker_hidden (Talker-wide tables, 2048 x 2048 in
 * "rightkit-qts 0.2.3 - Qwen3-TTS 1.7B -> QTS GGUF", section "Expected
 * verification shapes": each step's input then passes through
 * small_to_mtp like H and E0[q0], one more projection GEMM per step); hidden, ffn,
 * talker_hidden and vocab multiples of 128; 1 <= n_steps <= 15. */
typedef struct qp_geometry {
  int hidden, layers, n_q_heads, n_kv_heads, head_dim, ffn, vocab, n_steps;
  int talker_hidden, code_embed_dim, q0_vocab;
  float rms_eps, rope_theta;
} qp_geometry;

/* One weight tensor handed to qp_load_weights.
 * name:   the predictor-file name, e.g. "code_pred.blk.3.ffn_up.weight",
 *         "code_pred.small_to_mtp_projection.bias",
 *         "code_pred.codec_embd.7.weight", "code_pred.lm_head.0.weight",
 *         or "talker.codec_embd.weight" (the q0 table).
 * dtype:  matrices accept QP_BF16, QP_F16 or QP_Q8_0.  The projection and
 *         layer matrices (attn_q/k/v/output, ffn_gate/up/down) share one
 *         format, 16-bit (f16 and bf16 may mix) or Q8_0; the lm-heads share
 *         one, which may be 16-bit over Q8_0 matrices (the exporter's
 *         layout) but not Q8_0 over 16-bit ones.  Embedding tables (the
 *         code tables and the q0 table) accept QP_BF16 or QP_F16, one
 *         encoding for all of them; vectors (norms, bias) QP_F32.  A
 *         combination outside these is QP_ERR_WEIGHT_DTYPE.  A Q8_0
 *         matrix is kept twice on the device: as its blocks (the tile
 *         engine dequantises them on chip) and as two f16 images, hi =
 *         f16(d*q) and lo = f16(d*q - hi), for the small-batch and cluster
 *         engines (4 more bytes per weight); hi + lo = d*q exactly for
 *         d >= 2^-14.
 * dev_ptr: device memory, row-major HF layout [shape[0], shape[1]]; a Q8_0
 *         tensor is its raw block stream, shape[0] rows of shape[1]/32
 *         blocks.  Vectors use shape = {n, 0}. */
typedef struct qp_weight {
  const char* name;
  qp_dtype dtype;
  const void* dev_ptr;
  int64_t shape[2];
} qp_weight;

/* Sampling: z = logits / temperature; the top_k largest z (ties by lower
 * index) form the candidate set; the code is argmax over it of
 * z + gumbel[b, step, i], lowest index on ties.  gumbel is a device array
 * [B, n_steps, vocab] f32 of standard Gumbel noise supplied by the caller. */
typedef struct qp_sampling {
  float temperature;   /* > 0 */
  int top_k;           /* 1 .. vocab */
  const float* gumbel; /* device, [B, n_steps, vocab] */
} qp_sampling;

typedef struct qp_handle qp_handle;
typedef void* qp_stream;

/* Library ABI version (QP_ABI_VERSION). */
int qp_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* qp_status_string(qp_status s);

/* Fill *g with the default geometry.  QP_ERR_ARG if g is NULL. */
qp_status qp_default_geometry(qp_geometry* g);

/* Create a handle on the current CUDA device for batches of up to
 * max_batch frames (1 <= max_batch <= 65536).  Allocates the library-owned
 * scratch (activations, KV cache, status word) sized for max_batch.  On
 * error *out is set to NULL. */
qp_status qp_create(const qp_geometry* g, int max_batch, qp_handle** out);

/* Copy and repack the n weight tensors into library-owned device memory, on
 * stream s.  All 89 tensors must be supplied exactly once (the 88 of the
 * predictor file plus talker.codec_embd.weight); a missing, duplicate,
 * unknown, mis-shaped or wrongly typed tensor fails the whole load and
 * nothing is enqueued.  The caller may free its buffers once s has reached
 * this point.  May be called again to replace all weights. */
qp_status qp_load_weights(qp_handle* h, const qp_weight* w, int n, qp_stream s);

/* Greedy prediction for B frames (1 <= B <= max_batch), enqueued on s.
 *   H          device, [B, talker_hidden] f32, row-major, 16-byte aligned
 *   q0         device, [B] int32 in [0, q0_vocab)
 *   out_codes  device, [B, n_steps] int32: q1..q15 per frame
 *   out_logits device, [B, n_steps, vocab] f32, 16-byte aligned, or NULL to skip
 * int32 and f32 arrays must be 4-byte aligned; a misaligned pointer is
 * QP_ERR_ARG. */
qp_status qp_predict_frames(qp_handle* h, int B, const float* H, const int32_t* q0,
                            int32_t* out_codes, float* out_logits, qp_stream s);

/* As qp_predict_frames, plus:
 *   samp          NULL for greedy, else Gumbel top-k sampling (above)
 *   forced_codes  NULL, or device [B, n_steps] int32: teacher forcing.  The
 *                 input of step k+1 embeds forced_codes[b, k-1] instead of
 *                 the decided code; out_codes still holds the decisions. */
qp_status qp_predict_frames_ex(qp_handle* h, int B, const float* H, const int32_t* q0,
                               int32_t* out_codes, float* out_logits,
                               const qp_sampling* samp, const int32_t* forced_codes,
                               qp_stream s);

/* Host-buffer variant: H_host [B, talker_hidden] f32, q0_host [B] int32 and
 * codes_host [B, n_steps] int32 are host memory (pinned or pageable).
 * Copies the inputs to library-owned device buffers, predicts (greedy, or
 * sampling with a DEVICE gumbel array when samp is not NULL), copies the
 * codes back and synchronises s before returning. */
qp_status qp_predict_frames_host(qp_handle* h, int B, const float* H_host,
                                 const int32_t* q0_host, int32_t* codes_host,
                                 const qp_sampling* samp, qp_stream s);

/* Greedy prediction that allocates nothing, for callers that cannot let a
 * library call cudaMalloc for them: a process whose own allocator already
 * holds the GPU's memory, or a real-time audio path that forbids allocation
 * once it runs.  (The pages have no counterpart: this is a library
 * convenience, not part of the method.)  It runs the same kernel as
 * qp_predict_frames with the same arguments and outputs (no sampling, no
 * teacher forcing), but the kernel's scratch -- residual stream, tensor-core
 * operand, accumulators, logits, KV cache, barrier words -- lives in one
 * static device array of 8 MiB that every GPU loading the library holds
 * until the process exits.  Weights come from h, loaded beforehand; errors
 * the GPU detects still go to h's status word.
 *   - B must be at most 8, and the scratch B frames need under h's geometry
 *     must fit in 8 MiB (it does for the default geometry); otherwise
 *     QP_ERR_ARG and nothing is enqueued.
 *   - The first call on a device looks up the array's device address and
 *     sets the kernel's shared-memory limit; make that first call before any
 *     stream capture begins.
 *   - All calls share the one array and it keeps the last call's contents;
 *     the call clears the barrier words it needs at zero and writes every
 *     other byte before reading it.  Calls whose executions overlap on the
 *     GPU (other streams, other handles, other threads) race on the array:
 *     serialise them. */
qp_status qp_predict_frames_static(qp_handle* h, int B, const float* H, const int32_t* q0,
                                   int32_t* out_codes, float* out_logits, qp_stream s);

/* Deterministic mode, for callers that need run-to-run reproducibility
 * (the pages have no counterpart; a serving option, not part of the
 * method).  on != 0: later qp_predict_frames* calls on h give bit-identical
 * codes and logits for bit-identical inputs (same weights, handle geometry
 * and batch size).  Ordinarily the partial products of a weight matrix split
 * over several SMs meet in f32 atomic additions, whose order -- and so
 * whose last bits -- vary from run to run; a greedy or sampled code whose
 * margin is within that noise can then flip.  In this mode every output
 * tile's whole reduction runs on one SM (tensor-core accumulators, in a
 * fixed order), each output element receives exactly one addition, and the
 * rows' squared norms are summed from per-tile partial sums in tile order.
 * The calls run on the tile engine and cost more time at small batches,
 * where fewer SMs share each GEMM.  The state-slot calls of qp_sched.h are
 * not covered.  on == 0 restores the default.  QP_ERR_ARG for a null
 * handle; a later call with QP_ENGINE_SMALL forced (qp_debug.h) is
 * QP_ERR_ARG. */
qp_status qp_set_deterministic(qp_handle* h, int on);

/* Synchronise s, read and clear the device status word: QP_OK, or the
 * first device-detected error since the last read. */
qp_status qp_get_device_status(qp_handle* h, qp_stream s);

/* Number of GPU kernel launches one qp_predict_frames_ex call with these
 * arguments enqueues (for launch accounting); -1 on bad arguments. */
int qp_launches_per_call(qp_handle* h, int B, int sampling);

/* Frame-feedback embeddings: out[b][j] = E_j[codes[b][j]] as f32, for j =
 * 0 .. n_steps-1, where E_j is the loaded table code_pred.codec_embd.j
 * (bf16, converted exactly) and codes[b][j] is the frame's code q_{j+1} as
 * qp_predict_frames returns it ([B][n_steps] int32, device).  These are the
 * vectors of a frame's residual codes in the predictor's own embedding
 * space, table n_steps-1 included, which the loop itself never reads
 * (reading: the pages name the tables but not this use; it is inferred from
 * table 14's existence, "rightkit-qts 0.2.3", section "Loader contract").
 * out is [B][n_steps][code_embed_dim] f32, device, 16-byte aligned.  A code outside
 * [0, vocab) is clamped for addressing and latches QP_ERR_BAD_TOKEN in the
 * device status word.  QP_ERR_STATE if no weights are loaded, QP_ERR_ARG for
 * B < 0, null or misaligned pointers; B == 0 enqueues nothing. */
qp_status qp_code_embeddings(qp_handle* h, int B, const int32_t* codes, float* out, qp_stream s);

/* Free everything the handle owns (synchronises the device first). */
void qp_destroy(qp_handle* h);

#ifdef __cplusplus
}
#endif
#endif /* QP_H */
