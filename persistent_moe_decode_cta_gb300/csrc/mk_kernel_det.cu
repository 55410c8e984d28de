// The megakernel with deterministic layer accumulators (64-bit fixed-point sums whose
// value does not depend on the order of the adds), in namespace mk_det: the same source
// compiled with MK_DET = 1 (see mk_kernel.cu).
#define MK_DET 1
#include "mk_kernel.cu"
