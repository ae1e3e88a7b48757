/*
 * qp_gguf.h -- loading the Code Predictor's weights from GGUF files (libqp).
 *
 * The exporter of "rightkit-qts 0.2.3 - Qwen3-TTS 1.7B -> QTS GGUF" writes
 * the predictor into its own GGUF file, with the tensors
 * code_pred.small_to_mtp_projection.{weight,bias}, code_pred.output_norm,
 * code_pred.blk.{0..4}.* and code_pred.codec_embd / lm_head.{0..14}, and its
 * geometry as the metadata keys qwen3-tts.code_pred.{embedding_length,
 * attention.key_length, attention.head_count, attention.head_count_kv,
 * feed_forward_length, layer_count, vocab_size,
 * attention.layer_norm_rms_epsilon, rope.freq_base} (sections "Loader
 * contract" and "Expected verification shapes").  The q0 table,
 * talker.codec_embd.weight, lives in the Talker's file.  Vectors are F32,
 * embeddings and output heads F16, eligible matrices Q8_0 (section
 * "Upstream differences & verification scope"); tensor dimensions are
 * stored in GGML order (innermost first) and are reversed here to the HF
 * [out, in] order qp_load_weights uses.
 *
 * Files are GGUF version 2 or 3, little-endian: header, metadata key/values,
 * tensor table, then the tensor data, each tensor at its offset from the
 * start of the data section, which begins at the next multiple of
 * general.alignment (32 when absent) after the table.  Tensor types read:
 * F32, F16, BF16 and Q8_0 (blocks of {f16 d; int8 q[32]} along the
 * innermost dimension); any other type fails the load with
 * QP_ERR_WEIGHT_DTYPE.
 *
 * Everything here is host code: qp_gguf_open and the queries read the file
 * only (no CUDA call); qp_gguf_load_weights stages the needed tensors
 * through pinned host memory to temporary device buffers, calls
 * qp_load_weights on `stream`, synchronises the stream and frees them.
 */
#ifndef QP_GGUF_H
#define QP_GGUF_H

#include <stdint.h>

#include "qp.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct qp_gguf qp_gguf;

/* Parse the header, metadata and tensor table of the GGUF file at `path`.
 * QP_ERR_ARG for null arguments, an unreadable file, a bad magic, an
 * unsupported version or a truncated or inconsistent table (a tensor whose
 * data would lie past the end of the file); *out is NULL then. */
qp_status qp_gguf_open(const char* path, qp_gguf** out);
void qp_gguf_close(qp_gguf* f);

int qp_gguf_tensor_count(const qp_gguf* f);
/* Tensor i: its name (owned by f), storage type and HF-order shape
 * (shape[1] = 0 for a vector).  QP_ERR_ARG for a bad index, or for a tensor
 * of more than two dimensions; *dtype is set to -1 when the type is not one
 * of the four read here. */
qp_status qp_gguf_tensor_info(const qp_gguf* f, int i, const char** name, int* dtype, int64_t shape[2]);

/* Predictor geometry: the qwen3-tts.code_pred.* keys of `predictor` where
 * present; talker_hidden and code_embed_dim from the projection's and
 * table 0's input widths, n_steps from the number of lm-heads, q0_vocab
 * from talker.codec_embd.weight in `talker` (or in `predictor`; may be
 * NULL if the table is in the predictor file).  QP_ERR_WEIGHT_MISSING if a
 * tensor it needs is absent, QP_ERR_WEIGHT_SHAPE if the keys and the tensor
 * shapes disagree. */
qp_status qp_gguf_geometry(const qp_gguf* predictor, const qp_gguf* talker, qp_geometry* g);

/* Load the predictor's 89 tensors, each found by name in the first of the
 * n_files files that holds it (other tensors are ignored), into h through
 * qp_load_weights.  Its statuses pass through (a tensor missing from every
 * file is QP_ERR_WEIGHT_MISSING); QP_ERR_ARG if a file cannot be read;
 * QP_ERR_OOM if the staging buffers cannot be allocated. */
qp_status qp_gguf_load_weights(qp_handle* h, const qp_gguf* const* files, int n_files, qp_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* QP_GGUF_H */
