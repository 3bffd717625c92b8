// Kernel instantiations for head dimension 128.
#include "santa_cluster.cuh"
#include "santa_dense.cuh"
#include "santa_gather.cuh"
#include "santa_kernels.h"
#include "santa_score.cuh"

namespace santa {

const void *kernel_d128(int kind, int G)
{
    if (kind == KIND_GATHER) {
        switch (G) {
        case 1: return (const void *)santa_gather_kernel<128, 1>;
        case 2: return (const void *)santa_gather_kernel<128, 2>;
        case 4: return (const void *)santa_gather_kernel<128, 4>;
        case 8: return (const void *)santa_gather_kernel<128, 8>;
        }
        return nullptr;
    }
    if (kind == KIND_CLUSTER) {  // the single-pass kernel for small batches (thread-block clusters)
        switch (G) {
        case 1: return (const void *)santa_cluster_kernel<128, 1>;
        case 2: return (const void *)santa_cluster_kernel<128, 2>;
        case 4: return (const void *)santa_cluster_kernel<128, 4>;
        case 8: return (const void *)santa_cluster_kernel<128, 8>;
        }
        return nullptr;
    }
    if (kind == KIND_DMERGE) return (const void *)santa_dense_merge_kernel<128>;
    if (kind == KIND_SCORE) {
        switch (G) {
        case 1: return (const void *)santa_score_kernel<128, 1>;
        case 2: return (const void *)santa_score_kernel<128, 2>;
        case 4: return (const void *)santa_score_kernel<128, 4>;
        case 8: return (const void *)santa_score_kernel<128, 8>;
        }
    } else if (kind == KIND_DENSE) {
        switch (G) {
        case 1: return (const void *)santa_dense_kernel<128, 1>;
        case 2: return (const void *)santa_dense_kernel<128, 2>;
        case 4: return (const void *)santa_dense_kernel<128, 4>;
        case 8: return (const void *)santa_dense_kernel<128, 8>;
        }
    }
    return nullptr;
}

}  // namespace santa
