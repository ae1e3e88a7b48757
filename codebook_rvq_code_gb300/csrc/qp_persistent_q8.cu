// The tile engine's kernel for Q8_0 matrices: the program of qp_persistent.cu
// compiled a second time with the four dequantising warps in.
#define QP_TILE_Q8 1
#include "qp_persistent.cu"
