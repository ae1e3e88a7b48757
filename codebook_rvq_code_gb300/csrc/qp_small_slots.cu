// The small-batch engine's state-slot kernel (include/qp_sched.h): the same
// program and sections as the frame-loop kernel in qp_small.cu, compiled a
// second time for calls whose rows keep their KV state in slots between
// calls and may stand at different steps.
#define QP_SMALL_SLOTS 1
#include "qp_small.cu"
