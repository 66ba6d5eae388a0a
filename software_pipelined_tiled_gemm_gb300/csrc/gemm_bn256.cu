// Kernel instance: 128 x 256 output tiles.
#include "gemm_instance.cuh"
SPGEMM_DEFINE_BN(256)
