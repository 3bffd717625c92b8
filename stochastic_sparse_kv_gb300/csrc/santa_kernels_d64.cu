// Kernel instantiations for head dimension 64.
#include "santa_dense.cuh"
#include "santa_kernels.h"

namespace santa {

const void *kernel_d64(int kind, int G)
{
    if (kind == KIND_SAMPLE) {
        switch (G) {
        case 1: return (const void *)santa_sample_kernel<64, 1>;
        case 2: return (const void *)santa_sample_kernel<64, 2>;
        case 4: return (const void *)santa_sample_kernel<64, 4>;
        case 8: return (const void *)santa_sample_kernel<64, 8>;
        }
    } else {
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
