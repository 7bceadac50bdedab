// The paired CTA shape of the kernel: two CTAs of 12 consumer warps per SM
// (12 KB staging chunks, 6144 candidates each). Same source as the wide
// shape, with its own constants, in namespace ltk::pair.
#define LTK_SHAPE_PAIR 1
#include "topk_kernel.cu"
