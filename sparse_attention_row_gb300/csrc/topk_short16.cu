// The short-row kernel with 16 warps per CTA (512 threads, 512 candidate slots
// per warp, the same 8192 candidates and 128 KB ring as the 32-warp instance),
// in namespace ltk::short16. Same source as ltk::shortrow.
#define LTK_SHORT_NS short16
#define LTK_SHORT_THREADS kShort16CtaThreads
#define LTK_SHORT_REGION 512
#include "topk_short.cu"
