// Two-CTA persistent tile 256x224 (cta_group::2), one translation unit.
#include "gemm_launch.cuh"
SDT_INSTANTIATE_GEMM_PAIR(224)
