// santa_kernels.h -- internal: kernel registry shared by the host API and the kernel
// translation units (one per head dimension).
#pragma once

namespace santa {

// KIND_GATHER + v: the value-stage kernel of variant v (GATHER_XD | GATHER_IID | GATHER_WIDE)
enum KernelKind : int { KIND_SCORE = 0, KIND_DENSE = 1, KIND_DMERGE = 3, KIND_CLUSTER = 4, KIND_GATHER = 8 };

// Kernel entry for (kind, G) at head dimension 64 or 128, or nullptr.
const void *kernel_d64(int kind, int G);
const void *kernel_d128(int kind, int G);

// Dynamic shared-memory bytes of the score, value-stage and dense kernels.
int score_smem_bytes(int D, int G, int B);
int gather_smem_bytes(int D, int G, int S, int nch_used, int mode, bool xdedup, int nth);
int dense_smem_bytes(int D, int G, int B);
int cluster_smem_bytes(int D, int G, int LW, int S, int mode, int C, int ns);

// Device points kernel (santa_sample_points).
const void *points_kernel();
const void *points_iid_kernel();

}  // namespace santa
