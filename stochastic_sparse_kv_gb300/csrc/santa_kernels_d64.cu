// Kernel instantiations for head dimension 64.
#include "santa_cluster.cuh"
#include "santa_dense.cuh"
#include "santa_gather.cuh"
#include "santa_kernels.h"
#include "santa_score.cuh"

namespace santa {

const void *kernel_d64(int kind, int G)
{
    if (kind >= KIND_GATHER && kind < KIND_GATHER + 8) {  // (group dedup: G > 1, narrow team)
        const int v = kind - KIND_GATHER;
        switch (G * 8 + v) {
        case 8: return (const void *)santa_gather_kernel<64, 1, 0>;
        case 10: return (const void *)santa_gather_kernel<64, 1, GATHER_IID>;
        case 12: return (const void *)santa_gather_kernel<64, 1, GATHER_WIDE>;
        case 14: return (const void *)santa_gather_kernel<64, 1, GATHER_IID | GATHER_WIDE>;
        case 16: return (const void *)santa_gather_kernel<64, 2, 0>;
        case 17: return (const void *)santa_gather_kernel<64, 2, GATHER_XD>;
        case 18: return (const void *)santa_gather_kernel<64, 2, GATHER_IID>;
        case 19: return (const void *)santa_gather_kernel<64, 2, GATHER_XD | GATHER_IID>;
        case 20: return (const void *)santa_gather_kernel<64, 2, GATHER_WIDE>;
        case 22: return (const void *)santa_gather_kernel<64, 2, GATHER_IID | GATHER_WIDE>;
        case 32: return (const void *)santa_gather_kernel<64, 4, 0>;
        case 33: return (const void *)santa_gather_kernel<64, 4, GATHER_XD>;
        case 34: return (const void *)santa_gather_kernel<64, 4, GATHER_IID>;
        case 35: return (const void *)santa_gather_kernel<64, 4, GATHER_XD | GATHER_IID>;
        case 36: return (const void *)santa_gather_kernel<64, 4, GATHER_WIDE>;
        case 38: return (const void *)santa_gather_kernel<64, 4, GATHER_IID | GATHER_WIDE>;
        case 64: return (const void *)santa_gather_kernel<64, 8, 0>;
        case 65: return (const void *)santa_gather_kernel<64, 8, GATHER_XD>;
        case 66: return (const void *)santa_gather_kernel<64, 8, GATHER_IID>;
        case 67: return (const void *)santa_gather_kernel<64, 8, GATHER_XD | GATHER_IID>;
        case 68: return (const void *)santa_gather_kernel<64, 8, GATHER_WIDE>;
        case 70: return (const void *)santa_gather_kernel<64, 8, GATHER_IID | GATHER_WIDE>;
        }
        return nullptr;
    }
    if (kind == KIND_CLUSTER) {  // the single-pass kernel for small batches (thread-block clusters)
        switch (G) {
        case 1: return (const void *)santa_cluster_kernel<64, 1>;
        case 2: return (const void *)santa_cluster_kernel<64, 2>;
        case 4: return (const void *)santa_cluster_kernel<64, 4>;
        case 8: return (const void *)santa_cluster_kernel<64, 8>;
        }
        return nullptr;
    }
    if (kind == KIND_DMERGE) return (const void *)santa_dense_merge_kernel<64>;
    if (kind == KIND_SCORE) {
        switch (G) {
        case 1: return (const void *)santa_score_kernel<64, 1>;
        case 2: return (const void *)santa_score_kernel<64, 2>;
        case 4: return (const void *)santa_score_kernel<64, 4>;
        case 8: return (const void *)santa_score_kernel<64, 8>;
        }
    } else if (kind == KIND_DENSE) {
        switch (G) {
        case 1: return (const void *)santa_dense_kernel<64, 1>;
        case 2: return (const void *)santa_dense_kernel<64, 2>;
        case 4: return (const void *)santa_dense_kernel<64, 4>;
        case 8: return (const void *)santa_dense_kernel<64, 8>;
        }
    }
    return nullptr;
}

}  // namespace santa
