// Persistent tile 128x128 (double-buffered TMEM accumulator), one translation unit.
#include "gemm_launch.cuh"
SDT_INSTANTIATE_GEMM_PERSISTENT(128)
