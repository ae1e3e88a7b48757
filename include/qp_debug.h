/*
 * qp_debug.h -- phase tracing of libqp's persistent kernel (profiling aid).
 *
 * With tracing on, thread 0 of every CTA stamps the GPU global timer (ns)
 * when its consumer warps start and finish each section of the program (the
 * step-1 inputs, each GEMM's epilogues, each layer's attention, each step's
 * inputs and decisions, in program order).  A section's end includes its
 * waits for other CTAs' tiles.  Off by default; the stamps cost two global
 * stores per section.  Not part of the method.
 */
#ifndef QP_DEBUG_H
#define QP_DEBUG_H

#include <stdint.h>

#include "qp.h"

#ifdef __cplusplus
extern "C" {
#endif

/* enable != 0: allocate a device buffer for up to 8192 sections x the SM count
 * and record every later call into it (each call overwrites the last);
 * enable == 0: stop recording and free it.  Synchronises the device. */
qp_status qp_trace_enable(qp_handle* h, int enable);

/* Copy the last call's stamps to host memory: host[(section * n_cta + cta) * 2
 * + {0: start, 1: end}], for `phases` sections (at most the recorded ones).
 * When `phases` is 8192 (all of them), each CTA's event log follows: 16384
 * words per CTA, consumer events first, MMA-warp events from word 8192; a
 * word is (globaltimer ns mod 2^48) << 16 | event code << 12 | GEMM index,
 * zero where unused.  *n_cta receives the CTA count.  Synchronises the
 * device.  Returns the number of sections copied, or -1 if tracing is off or
 * an argument is bad. */
int qp_trace_read(qp_handle* h, uint64_t* host, int phases, int* n_cta);

#ifdef __cplusplus
}
#endif
#endif /* QP_DEBUG_H */
