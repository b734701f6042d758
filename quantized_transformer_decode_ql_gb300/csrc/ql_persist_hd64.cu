// Persistent decode step kernels for head_dim 64 (the kernel itself is in ql_persist.cuh).
#include "ql_persist.cuh"

namespace ql {
cudaError_t persist_dispatch_hd64(int G, bool launch, const PersistParams* p, size_t smem, int grid,
                                  cudaStream_t s, int* occ) {
    return persist::dispatch<64>(G, launch, p, smem, grid, s, occ);
}
}  // namespace ql
