// The small CTA shape of the kernel: 8 consumer warps, 8 KB staging chunks and
// 4096 candidates, about 83 KB of shared memory, for devices or partitions
// that cannot give a CTA the 113 KB of the paired shape. Same source as the
// other shapes, with its own constants, in namespace ltk::small.
#define LTK_SHAPE_SMALL 1
#include "topk_kernel.cu"
