/*
 * qp_rvq.h -- residual-vector-quantisation codebooks for the codec side of
 * the Code Predictor's output (libqp).
 *
 * The Code Predictor emits, per audio frame, the codes q0..q15 of a
 * residual vector quantiser: stage i quantises what the earlier stages left,
 * r_i = x - sum_{j<i} q_j ("拆解 Qwen3-TTS：OpenVINO 移植过程中的图分离与调度实践",
 * section 1, "RVQ 的层级逻辑"), so the codec's decoder starts from the sum of
 * the picked codebook vectors, x^ = sum_i C_i[code_i].  The codebooks are
 * stored EMA-trained, as a running sum of assigned vectors and a per-entry
 * usage count, and the codebook is their ratio,
 * C = embedding_sum / (cluster_usage + 1e-7) ("Qwen3-TTS на Rust", section
 * "Проблема 1: Формат codebook'ов").
 *
 * Layouts (row-major, f32, all device memory owned by the caller):
 *   embedding_sum, codebooks   [n_codebooks][codebook_size][dim]
 *   cluster_usage              [n_codebooks][codebook_size]
 *   codes                      [n_frames][n_codebooks] int32 (code of stage i in column i)
 *   out                        [n_frames][dim]
 * dim must be a multiple of 4 and every pointer 16-byte aligned (the
 * kernels move 4 floats per access).  Both calls only enqueue work on
 * `stream`; host-detectable argument errors return before anything is
 * enqueued.  Results are exact with respect to f32 arithmetic: the division
 * is IEEE-rounded and the sum adds the stages in order 0, 1, ..., without
 * fused multiply-adds.
 */
#ifndef QP_RVQ_H
#define QP_RVQ_H

#include <stdint.h>

#include "qp.h"

#ifdef __cplusplus
extern "C" {
#endif

/* codebooks = embedding_sum / (cluster_usage + 1e-7), element by element
 * (codebooks may alias embedding_sum).  QP_ERR_ARG for null or misaligned
 * pointers, non-positive sizes or dim % 4 != 0; QP_ERR_CUDA if the launch
 * fails. */
qp_status qp_rvq_normalize(const float* embedding_sum, const float* cluster_usage, int n_codebooks,
                           int codebook_size, int dim, float* codebooks, qp_stream stream);

/* out[n] = sum_{i < n_codebooks} codebooks[i][codes[n][i]] for n < n_frames
 * (n_frames == 0 enqueues nothing).  A code outside [0, codebook_size) is
 * clamped for addressing and, if `status` is not NULL, QP_ERR_BAD_TOKEN is
 * stored into the device int *status (first error wins; the caller zeroes
 * it).  QP_ERR_ARG for null or misaligned pointers, negative n_frames,
 * non-positive sizes or dim % 4 != 0; QP_ERR_CUDA if the launch fails. */
qp_status qp_rvq_decode(const float* codebooks, int n_codebooks, int codebook_size, int dim,
                        const int32_t* codes, int n_frames, float* out, int* status, qp_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* QP_RVQ_H */
