// qmm_batch_mix.cu -- the batched-matmul kernel (qmm_batch.cuh) whose items
// carry their own weight types: Q8_0, Q4_0, Q5_0, Q4_K and Q6_K in any mix,
// as in the mixed-type files (Q4_K_M) the "GGUF 文件" page describes.
#include "qmm_internal.h"

namespace qmm {

cudaError_t launch_batch_mix(int am, BatchParams& p, int mt, int grid, int smem_max, cudaStream_t s) {
    return am == A_INT8 ? batch_go_mt<T_MIX, A_INT8>(p, mt, grid, smem_max, s)
                        : batch_go_mt<T_MIX, A_F32>(p, mt, grid, smem_max, s);
}

}  // namespace qmm
