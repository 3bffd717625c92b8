// santa_sample.cuh -- building blocks of the SANTA decode kernels, sm_103a.
//
// "Stochastic Sparse Attention for Memory-Bound Inference" (abstract): the score stage
// reads all n_k keys and forms the post-softmax distribution; the value stage samples
// S << n_k indices from it (stratified or systematic sampling) and gather-adds only
// those V rows, scaled by 1/S.  The score stage is santa_score_kernel
// (santa_score.cuh), the value stage santa_gather_kernel (santa_gather.cuh); this file
// holds the pieces they and the dense kernel share: the per-tile grouped-query dot
// products, the error-free re-scoring of heavy keys, the work-item space and small
// block-level helpers.
#pragma once

#include "santa_common.cuh"

namespace santa {

template <int D, int G>
struct SampleCfg {
    static constexpr int P = D / 16;            // lanes per key in the score loop
    static constexpr int KW = 64 / P;           // keys per warp and tile (2 per lane group)
    static constexpr int TK = NWARP * KW;       // keys per tile
    static constexpr int ROWB = 2 * D;          // bytes per K row
    static constexpr int NSTAGE = 4;
    static constexpr int V = 2 * G;             // partial dots per lane
    static constexpr int NV = V >= P ? V / P : 1;   // scores per lane after the reduction
    static constexpr int REP = V >= P ? 1 : P / V;  // lanes holding the same score
    static constexpr int EPL = D / 32;          // V elements per lane in the gather
    static_assert(TK * ROWB == TILE_BYTES, "tile size");
    static_assert(LMIN % TK == 0, "split length must be a multiple of the tile");

    __host__ __device__ static constexpr int vidx(int sub, int i) { return V >= P ? sub * NV + i : sub / REP; }
    __host__ __device__ static constexpr int head_of(int lane, int i) { return vidx(lane % P, i) % G; }
    __host__ __device__ static constexpr int key2_of(int lane, int i) { return vidx(lane % P, i) / G; }
    // Flipping lane bit m leaves the heads of every score slot unchanged.
    __host__ __device__ static constexpr bool same_heads(int m)
    {
        for (int l = 0; l < 32; ++l)
            for (int i = 0; i < NV; ++i)
                if (head_of(l ^ m, i) != head_of(l, i)) return false;
        return true;
    }
    __host__ __device__ static constexpr unsigned same_mask()
    {
        unsigned r = 0;
        for (int m = 1; m < 32; m <<= 1)
            if (same_heads(m)) r |= (unsigned)m;
        return r;
    }
    // Lane-xor masks (as a bit set) that keep every score slot's head: evaluated by the
    // compiler, so the per-tile reductions below unroll to a fixed shuffle sequence.
    static constexpr unsigned SAME = same_mask();
};

__host__ __device__ inline int next_pow2(int x)
{
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

// Descriptor of a staged tile (int4: group b*H_kv+g, (unit << 8) | tile, rows, flags).
enum : int { DESC_END = -1 };
// Flags: the tile is the first of a new (b, g), whose query heads come in staging buffer
// (flags >> TF_QB_SHIFT) & 1, or must be read from global memory; the tile is the last
// of its work unit.
enum : int { TF_NEWQ = 1, TF_QGLOBAL = 2, TF_QB_SHIFT = 2, TF_LAST = 8 };

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

// Reduce-scatter of the V partial dots of a lane group of P lanes: after it the lane
// keeps the sums of the value slots given by SampleCfg::vidx.
template <int M, int C, int V>
__device__ __forceinline__ void rs_step(float (&val)[V], int sub)
{
    if constexpr (M >= 1) {
        if constexpr (C > 1) {
            constexpr int H = C / 2;
            const bool up = (sub & M) != 0;
#pragma unroll
            for (int i = 0; i < H; ++i) {
                const float send = up ? val[i] : val[i + H];
                const float recv = __shfl_xor_sync(0xffffffffu, send, M);
                val[i] = __fadd_rn(up ? val[i + H] : val[i], recv);
            }
            rs_step<M / 2, H, V>(val, sub);
        } else {
            val[0] = __fadd_rn(val[0], __shfl_xor_sync(0xffffffffu, val[0], M));
            rs_step<M / 2, 1, V>(val, sub);
        }
    }
}

// fp32 dots of 2 keys (rows kbase, kbase+1 of the tile) with the G query heads; lane
// sub of the group holds 16 elements: 16-byte chunks sub and sub + P of each row.
template <int D, int G>
__device__ __forceinline__ void tile_dots(const uint8_t *tile, int kbase, int sub,
                                          const unsigned long long (&qp)[G][8], float (&val)[2 * G])
{
    using C = SampleCfg<D, G>;
    unsigned long long acc[2][G];
#pragma unroll
    for (int kk = 0; kk < 2; ++kk)
#pragma unroll
        for (int h = 0; h < G; ++h) acc[kk][h] = 0ull;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
        const uint8_t *row = tile + (kbase + kk) * C::ROWB;
        const uint4 a = *reinterpret_cast<const uint4 *>(row + 16 * sub);
        const uint4 c = *reinterpret_cast<const uint4 *>(row + 16 * (sub + C::P));
        const uint32_t wv[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const unsigned long long kp = bf16x2_to_f32x2(wv[i]);
#pragma unroll
            for (int h = 0; h < G; ++h) ffma2(acc[kk][h], qp[h][i], kp);
        }
    }
#pragma unroll
    for (int kk = 0; kk < 2; ++kk)
#pragma unroll
        for (int h = 0; h < G; ++h) val[kk * G + h] = f32x2_sum(acc[kk][h]);
    rs_step<C::P / 2, 2 * G, 2 * G>(val, sub);
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

// ------------------------------------------------------------------ block helpers

// Exclusive block scan of one int per thread; returns the block total via *total.
__device__ __forceinline__ int block_excl_scan(int v, int *scratch /*NWARP+1 ints*/, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int w = 0; w < NWARP; ++w) {
            const int t = scratch[w];
            scratch[w] = acc;
            acc += t;
        }
        scratch[NWARP] = acc;
    }
    __syncthreads();
    const int res = scratch[warp] + x - v;
    *total = scratch[NWARP];
    __syncthreads();
    return res;
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



// misc[] words of a kernel's shared block
enum : int { MISC_SCAN = 0 /* NWARP+1 words */, MISC_LAST = 12 };

// Work items of a call: per batch row b, H_kv * ceil(n_b / L) splits (H_kv items when
// n_b = 0).  Fills nb[b] (clamped lengths) and the exclusive prefix prefix[0..B] of the
// item counts; flags out-of-range lengths.  Called by every thread of the CTA.
__device__ __forceinline__ void build_item_space(const Params &p, int *nb, int *prefix, int *misc)
{
    constexpr int PER = (BMAX + NT - 1) / NT;
    const int tid = threadIdx.x;
    int cnt[PER];
    int local = 0;
    bool bad = false;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int b = tid * PER + i;
        cnt[i] = 0;
        if (b < p.B) {
            int n = p.seq_lens[b];
            if (n < 0 || n > p.n_max) {
                bad = true;
                n = 0;
            }
            nb[b] = n;
            cnt[i] = p.H_kv * (n > 0 ? (n + p.L - 1) / p.L : 1);
            local += cnt[i];
        }
    }
    if (bad && blockIdx.x == 0) set_dev_error(p.ctrl, DEV_BAD_SEQLEN);
    int total;
    int run = block_excl_scan(local, misc + MISC_SCAN, &total);
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int b = tid * PER + i;
        if (b < p.B) prefix[b] = run;
        run += cnt[i];
    }
    if (tid == 0) prefix[p.B] = total;
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
