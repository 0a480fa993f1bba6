// The sampling kernels for ARC_F16 logits, without a token history.
#include "kernel_set_impl.cuh"

template struct arc::KernelSet<ARC_F16, false>;
