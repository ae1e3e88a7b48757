/*
 * qp_sched.h -- ragged-step batching for a frame scheduler (libqp).
 *
 * The serving stack of "テキスト音声合成モデルを50ミリ秒未満で応答させる方法"
 * (section "Qwen3-TTSの最適化方法", items 1 and 2) puts the Talker, the Code
 * Predictor and the codec under one scheduler that batches requests waiting
 * for the same module, keeps work units short so that urgent requests can
 * be interleaved, and fills a batch around an urgent request with
 * compatible work.  A scheduler that stops a frame between steps and
 * refills the batch needs calls whose rows are at different steps.  These
 * entry points give it that: a frame's state (its KV cache, positions
 * 0..k) lives in one of the handle's max_batch state slots between calls;
 * qp_begin_frames runs step 1 of new frames into their slots, and
 * qp_step_frames advances each of its rows by one step from the row's own
 * step, so one call may hold frames at steps 2, 7 and 15 together.  The
 * arithmetic is that of qp_predict_frames: a frame run through begin and
 * then steps 2..n_steps, feeding each step the code q_{k-1} it chose (or a
 * forced one), gets the codes and logits of qp_predict_frames.
 *
 * Served by the small-batch engine: any weight format qp_load_weights
 * accepts (Q8_0 matrices through their f16 hi + lo images), B <= 64 rows per call,
 * greedy decisions or Gumbel top-k sampling (the _ex calls).  A step call runs one step's layers over all its rows;
 * its output head holds one head matrix per distinct step among the rows
 * (the rows sorted into step groups), as one GEMM.  Slot and step arrays are HOST memory (a scheduler keeps
 * this bookkeeping on the host); the library sorts the rows by step and
 * stages the order to the device on `stream`.  Codes, logits and H/q0 are
 * device memory, in the caller's row order, aligned as for
 * qp_predict_frames (H and logits 16 bytes, int32 arrays 4).  Rows of one
 * call must name distinct slots.
 */
#ifndef QP_SCHED_H
#define QP_SCHED_H

#include <stdint.h>

#include "qp.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Step 1 of B new frames: positions 0 (H) and 1 (E0[q0]) into slots[b]'s KV
 * state, out_q1[b] = the frame's first residual code (device [B] int32),
 * out_logits [B][vocab] f32 (device, or NULL).  QP_ERR_ARG for a bad B, a
 * slot outside [0, max_batch), repeated slots, null pointers, or a handle
 * this path cannot serve (B > 64); QP_ERR_STATE without
 * weights.  Device errors latch in the status word as for
 * qp_predict_frames. */
qp_status qp_begin_frames(qp_handle* h, int B, const int32_t* slots, const float* H, const int32_t* q0,
                          int32_t* out_q1, float* out_logits, qp_stream stream);

/* One step for each of B frames: row b is at step steps[b] (2..n_steps) of
 * the frame in slots[b], whose state holds positions 0..steps[b]-1;
 * codes_in[b] (device int32) is the code q_{steps[b]-1} that enters as the
 * step's input; out_codes[b] (device) receives q_{steps[b]}, out_logits
 * [B][vocab] (device, or NULL) the step's logits.  The new position is
 * appended to the slot's state.  Errors as for qp_begin_frames, plus
 * QP_ERR_ARG for a step outside [2, n_steps]; an input code outside
 * [0, vocab) latches QP_ERR_BAD_TOKEN and is clamped. */
qp_status qp_step_frames(qp_handle* h, int B, const int32_t* slots, const int32_t* steps, const int32_t* codes_in,
                         int32_t* out_codes, float* out_logits, qp_stream stream);

/* As qp_begin_frames and qp_step_frames, but each row's code is drawn by
 * Gumbel top-k sampling (qp_sampling of qp.h: z = logits / temperature, the
 * top_k largest z, argmax of z + g) when samp is not NULL, greedy when it
 * is.  samp->gumbel is device [B][vocab] f32: row b's noise for the one step
 * this call decides for it, in the caller's row order.  A frame run through
 * these calls with the noise qp_predict_frames_ex would read for each of its
 * steps gets the same codes.  QP_ERR_ARG additionally for a temperature that
 * is not positive and finite, top_k outside [1, vocab], a null or
 * misaligned noise array, or a vocabulary above 4096. */
qp_status qp_begin_frames_ex(qp_handle* h, int B, const int32_t* slots, const float* H, const int32_t* q0,
                             int32_t* out_q1, float* out_logits, const qp_sampling* samp, qp_stream stream);
qp_status qp_step_frames_ex(qp_handle* h, int B, const int32_t* slots, const int32_t* steps, const int32_t* codes_in,
                            int32_t* out_codes, float* out_logits, const qp_sampling* samp, qp_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* QP_SCHED_H */
