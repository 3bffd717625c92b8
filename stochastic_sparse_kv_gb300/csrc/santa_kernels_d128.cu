// Kernel instantiations for head dimension 128.
#include "santa_cluster.cuh"
#include "santa_dense.cuh"
#include "santa_gather.cuh"
#include "santa_kernels.h"
#include "santa_score.cuh"

namespace santa {

const void *kernel_d128(int kind, int G)
{
    if (kind >= KIND_GATHER && kind < KIND_GATHER + 4) {  // (group dedup needs G > 1)
        const int v = kind - KIND_GATHER;
        switch (G * 4 + v) {
        case 4: return (const void *)santa_gather_kernel<128, 1, 0>;
        case 6: return (const void *)santa_gather_kernel<128, 1, GATHER_IID>;
        case 8: return (const void *)santa_gather_kernel<128, 2, 0>;
        case 9: return (const void *)santa_gather_kernel<128, 2, GATHER_XD>;
        case 10: return (const void *)santa_gather_kernel<128, 2, GATHER_IID>;
        case 11: return (const void *)santa_gather_kernel<128, 2, GATHER_XD | GATHER_IID>;
        case 16: return (const void *)santa_gather_kernel<128, 4, 0>;
        case 17: return (const void *)santa_gather_kernel<128, 4, GATHER_XD>;
        case 18: return (const void *)santa_gather_kernel<128, 4, GATHER_IID>;
        case 19: return (const void *)santa_gather_kernel<128, 4, GATHER_XD | GATHER_IID>;
        case 32: return (const void *)santa_gather_kernel<128, 8, 0>;
        case 33: return (const void *)santa_gather_kernel<128, 8, GATHER_XD>;
        case 34: return (const void *)santa_gather_kernel<128, 8, GATHER_IID>;
        case 35: return (const void *)santa_gather_kernel<128, 8, GATHER_XD | GATHER_IID>;
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
