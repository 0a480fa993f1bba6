// The sampling kernels for ARC_BF16 logits, without a token history.
#include "kernel_set_impl.cuh"

template struct arc::KernelSet<ARC_BF16, false>;
