// The batch > 1 instance of the persistent megakernel (tensor-core matvec tiles), compiled in a
// translation unit of its own: the device code is the same source (in a namespace of its own, so
// no symbol is defined twice), and the batch-1 kernels in mk_kernel.cu keep the inlining and
// register allocation they get alone.
#define MK_BATCHED_TU
#define mk mk_bat
#include "mk_kernel.cu"
