// Tensor-core path of the causal LLA forward pass (placeholder until the tcgen05 kernel lands).
#include <cuda_runtime.h>

#include "lla_internal.h"

namespace lla {

size_t tensor_workspace_bytes(int B, int H, int n, int d) {
    return (size_t)3 * B * H * n * d * 2 + 256;
}

cudaError_t launch_tensor(const Problem&, void*, cudaStream_t, const char** why) {
    *why = "tensor path not built";
    return cudaErrorNotSupported;
}

}  // namespace lla
