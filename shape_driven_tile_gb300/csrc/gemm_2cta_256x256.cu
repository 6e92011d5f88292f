// Two-CTA persistent tile 256x256 (cta_group::2), one translation unit.
#include "gemm_launch.cuh"
SDT_INSTANTIATE_GEMM_PAIR(256)
