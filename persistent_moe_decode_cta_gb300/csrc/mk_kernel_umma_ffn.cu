// The megakernel with the LM head and the bf16 expert / dense-FFN items on the tcgen05
// tensor cores (accumulators in tensor memory), in namespace mk_umma_ffn: the same source
// compiled with MK_UMMA = 2 (see mk_kernel.cu).
#define MK_UMMA 2
#include "mk_kernel.cu"
