// The megakernel with the LM head on the tcgen05 tensor cores (accumulator in tensor
// memory), in namespace mk_umma: the same source compiled with MK_UMMA = 1 (see
// mk_kernel.cu).
#define MK_UMMA 1
#include "mk_kernel.cu"
