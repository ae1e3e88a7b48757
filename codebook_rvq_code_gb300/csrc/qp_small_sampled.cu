// The small-batch engine's frame-loop kernel with Gumbel top-k sampling:
// the program and sections of qp_small.cu, compiled a second time with the
// sampling pass in, for calls with a temperature above zero.
#define QP_SMALL_SAMPLED 1
#include "qp_small.cu"
