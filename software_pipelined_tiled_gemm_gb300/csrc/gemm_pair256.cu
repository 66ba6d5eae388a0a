// Kernel instance: CTA pairs computing 256 x 256 output tiles.
#include "gemm_instance.cuh"
SPGEMM_DEFINE_PAIR(256)
