// santa_sample.cuh -- building blocks of the SANTA decode kernels, sm_103a.
//
// "Stochastic Sparse Attention for Memory-Bound Inference" (abstract): the score stage
// reads all n_k keys and forms the post-softmax distribution; the value stage samples
// S << n_k indices from it (stratified or systematic sampling) and gather-adds only
// those V rows, scaled by 1/S.  The score stage is santa_score_kernel
// (santa_score.cuh), the value stage santa_gather_kernel (santa_gather.cuh); this file
// holds the pieces they and the dense kernel share: the work-item space, the error-free
// re-scoring of heavy keys and small block-level helpers.
#pragma once

#include "santa_common.cuh"

namespace santa {

__host__ __device__ inline int next_pow2(int x)
{
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

// Marker of the end of the work in a staged-tile descriptor (int4; x = DESC_END).
enum : int { DESC_END = -1 };

struct Item {
    int b, g, r, n, ns;
};

__device__ __forceinline__ Item decode_item(int it, const int *prefix, const int *nb, int B, int H_kv, int L)
{
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= it) lo = mid; else hi = mid - 1;
    }
    Item x;
    x.b = lo;
    x.n = nb[lo];
    x.ns = x.n > 0 ? (x.n + L - 1) / L : 1;
    const int local = it - prefix[lo];
    x.g = local / x.ns;
    x.r = local % x.ns;
    (void)H_kv;
    return x;
}

// Error-free score of one K row (global memory) with query head qf (fp32 copies of the
// bf16 values, shared memory), by the four lanes of a quad (part = lane & 3: elements
// [D/4 part, D/4 (part+1))).  Products of two bf16 values are exact in fp32; two
// interleaved compensated sums per lane (Knuth's TwoSum, errors accumulated apart), then
// a TwoSum butterfly over the quad.  Every lane of the quad returns the score in log2
// units, s * scale * log2(e), as a normalised pair (hi, lo) accurate to about 2^-44
// relative.  All 32 lanes of the warp must call it (it shuffles).
template <int D>
__device__ __forceinline__ void rescore_key_quad(const uint16_t *krow, const float *qf, int part, float k2_hi,
                                                 float k2_lo, float &hi, float &lo)
{
    constexpr int NE = D / 4;  // elements per lane: 32 or 16
    const uint4 *k4 = reinterpret_cast<const uint4 *>(krow + NE * part);
    const float *qp = qf + NE * part;
    uint4 kv[NE / 8];
#pragma unroll
    for (int c = 0; c < NE / 8; ++c) kv[c] = __ldcg(k4 + c);
    float s0 = 0.f, e0 = 0.f, s1 = 0.f, e1 = 0.f, t;
#pragma unroll
    for (int c = 0; c < NE / 8; ++c) {
        const uint32_t wv[4] = {kv[c].x, kv[c].y, kv[c].z, kv[c].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int d0 = 8 * c + 2 * i;
            two_sum(s0, __fmul_rn(qp[d0], bf16lo_to_f32(wv[i])), s0, t);
            e0 = __fadd_rn(e0, t);
            two_sum(s1, __fmul_rn(qp[d0 + 1], bf16hi_to_f32(wv[i])), s1, t);
            e1 = __fadd_rn(e1, t);
        }
    }
    float s, e;
    two_sum(s0, s1, s, t);
    e = __fadd_rn(__fadd_rn(e0, e1), t);
#pragma unroll
    for (int m = 1; m <= 2; m <<= 1) {
        const float s2 = __shfl_xor_sync(0xffffffffu, s, m);
        const float e2 = __shfl_xor_sync(0xffffffffu, e, m);
        two_sum(s, s2, s, t);
        e = __fadd_rn(__fadd_rn(e, e2), t);
    }
    fast_two_sum(s, e, s, e);
    // (s + e) * (k2_hi + k2_lo) to about 2^-46 relative
    const float P = __fmul_rn(s, k2_hi);
    float E = __fmaf_rn(s, k2_hi, -P);
    E = __fmaf_rn(s, k2_lo, E);
    E = __fmaf_rn(e, k2_hi, E);
    fast_two_sum(P, E, hi, lo);
}

// ------------------------------------------------------------------ search helpers

// The key of a chunk that a target selects: the first k whose running sum of the chunk's
// weights (fp32, added in key order) exceeds the target's remainder r inside the chunk.
// The running sum never decreases, so that k is the number of running sums <= r -- two
// instructions a key instead of a branch.  When there is none (rounding put the target
// past the chunk's mass) it is the chunk's last key of positive weight.
__device__ __forceinline__ int chunk_pick(const float (&wv)[CHUNK], int jn, float r)
{
    float P = 0.f;
    int cnt = 0;
#pragma unroll
    for (int k = 0; k < CHUNK; ++k) {
        P = __fadd_rn(P, k < jn ? wv[k] : 0.f);
        cnt += (P <= r) ? 1 : 0;
    }
    if (cnt < CHUNK) return cnt;
    int last = 0;
#pragma unroll
    for (int k = 0; k < CHUNK; ++k)
        if (k < jn && wv[k] > 0.f) last = k;
    return last;
}

__device__ __forceinline__ int lower_bound_i(const int *a, int n, int key)
{
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] < key) lo = mid + 1; else hi = mid;
    }
    return lo;
}

__device__ __forceinline__ int upper_bound_i(const int *a, int n, int key)
{
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] <= key) lo = mid + 1; else hi = mid;
    }
    return lo;
}
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace santa
