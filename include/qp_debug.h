/*
 * qp_debug.h -- engine selection and phase tracing of libqp's persistent
 * kernels (profiling and testing aids; not part of the method).
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

/* The frame loop has three schedules of the same computation.  Two split
 * every weight matrix into (128-row tile, 128-column K slice) units spread
 * over all SMs.  The tile engine serves any batch and both weight formats: a
 * completed tile is finished (residual, norm, SwiGLU, f16 operand) once by
 * the CTA whose partial completed it.  The small-batch engine serves both
 * formats too (Q8_0 matrices as their f16 hi + lo images, two slices per
 * unit) with at most 64 frames per call: partials go straight into their
 * destination and each consumer builds its operand slice from it, which
 * removes one dependent global round trip per GEMM.  The cluster engine
 * serves greedy calls of at most 32 frames, for geometries with head_dim
 * 128, two q heads per kv head, a hidden size of 512 or 1024, an FFN size a
 * multiple of 256, a vocabulary a multiple of 512 and
 * at most 7 layers (the 1.7B predictor's: the KV cache of a CTA's frames
 * stays in its tensor memory), with 16-bit or Q8_0 matrices (Q8_0 through their
 * f16 hi + lo images) and code tables as wide as the hidden size or as the
 * Talker state (then projected at every step): one 8-CTA thread-block cluster per kv head runs
 * QKV, attention and O, one per 256 FFN columns gate/up, SwiGLU and down,
 * partial products meeting in the cluster's shared memory, so a layer has two
 * grid-wide dependencies instead of five.  QP_ENGINE_AUTO (the default) takes
 * the cluster engine where it serves the call, else the small-batch engine
 * for calls of at most 40 frames, else the tile engine: the order of their
 * speed on GB300. */
typedef enum {
  QP_ENGINE_AUTO = 0,
  QP_ENGINE_TILE = 1,
  QP_ENGINE_SMALL = 2,
  QP_ENGINE_CLUSTER = 3
} qp_engine;

/* The cluster engine is launched cooperatively (all clusters co-resident
 * or the launch fails).  Nsight Compute rejects a cooperative launch with a
 * cluster dimension; with the environment variable QP_CLUSTER_NO_COOP=1 set
 * when the library is first used, the engine is launched without the
 * cooperative attribute (the grid is still the number of clusters that fit
 * at once, every wait stays bounded, and a cluster's CTAs are always
 * scheduled together), so the profiler can capture it. */

/* Select the engine for later calls on h.  A call the selected engine cannot
 * serve returns QP_ERR_ARG: with QP_ENGINE_SMALL more than 64 frames,
 * sampling over a vocabulary above 4096, or the deterministic schedule; with
 * QP_ENGINE_CLUSTER anything outside the calls and geometries above (or the
 * deterministic schedule).  QP_ERR_ARG for a null handle or an unknown
 * engine. */
qp_status qp_set_engine(qp_handle* h, int engine);

/* Testing aid for the device-side failure path.  Every wait inside the
 * frame-loop kernels (on another CTA's counter, on a shared-memory barrier)
 * is bounded; one that runs out latches QP_ERR_TIMEOUT in the status word
 * and raises an abort flag that every other wait honours, so all CTAs
 * unwind -- copies and MMAs in flight retire, TMEM is freed -- and the
 * kernel returns.  Nothing traps.
 *   wait_limit_us > 0: the limit of each wait in later calls on h, in
 *     microseconds of SM clock; 0 restores the default (about one second).
 *   withhold_gemm >= 0: in later frame-loop calls on h, the CTA whose share
 *     of that GEMM of the program starts at its first unit leaves its first
 *     completion count out, so the GEMM's consumers wait until the limit
 *     runs out.  The program's GEMMs are numbered in order: 0 is step 1's
 *     projection, then each step's GEMMs (4 per layer: QKV, O, gate/up,
 *     down; then the head).  The cluster engine, whose program is not a
 *     list of GEMMs, takes any withhold_gemm >= 0 to mean: its first CTA
 *     leaves out its count of step 1, layer 0's attention job, so every MLP
 *     job waits until the limit runs out.  -1 (the default) turns it off.
 * QP_ERR_ARG for a null handle, wait_limit_us < 0 or withhold_gemm < -1. */
qp_status qp_debug_waits(qp_handle* h, int wait_limit_us, int withhold_gemm);

/* Tracing is compiled in only when libqp is built with QP_TRACE=1 in the
 * environment (codebook_rvq_code_gb300/build.py): the hooks sit on the
 * loop's critical path.  Without them, enable != 0 returns QP_ERR_STATE.
 *
 * enable != 0: allocate a device buffer for up to 8192 sections x the SM count
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
