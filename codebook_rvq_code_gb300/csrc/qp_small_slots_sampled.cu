// The small-batch engine's state-slot kernel with Gumbel top-k sampling
// (include/qp_sched.h, qp_begin_frames_ex / qp_step_frames_ex): the program
// and sections of qp_small.cu, compiled with both the state-slot calls and
// the sampling pass in, for state-slot calls with a temperature above zero.
#define QP_SMALL_SLOTS 1
#define QP_SMALL_SAMPLED 1
#include "qp_small.cu"
