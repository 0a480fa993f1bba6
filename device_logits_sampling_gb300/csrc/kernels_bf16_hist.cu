// The sampling kernels for ARC_BF16 logits, with a token history.
#include "kernel_set_impl.cuh"

template struct arc::KernelSet<ARC_BF16, true>;
