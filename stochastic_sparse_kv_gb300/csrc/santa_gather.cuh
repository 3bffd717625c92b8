// santa_gather.cuh -- SANTA value stage: sample points, CDF search, gather-add, sm_103a.
//
// "Stochastic Sparse Attention for Memory-Bound Inference" (abstract): sample S << n_k
// indices from the post-softmax distribution and aggregate only those value rows,
// scaled by 1/S.  One CTA per (batch row b, query head h), launched as a programmatic
// dependent of the score kernel (its point generation overlaps the score kernel's
// tail).  It
//   1. merges the split totals exactly: O_r = sum_{r'<r} W_r' 2^(c_r' - C), Z = O_ns;
//   2. draws the S sorted points t_s (systematic, stratified, or sorted iid) and maps
//      each to i_s = min{ j : C_j > t_s } by a split -> chunk -> key search;
//   3. gather-adds each distinct sampled V row once, weighted by its count, and
//      writes out = sum / S and the sorted indices.
#pragma once

#include "santa_sample.cuh"

namespace santa {

struct GatherSmem {
    int O, cr, idx, lead, acc, misc, total;
};

__host__ __device__ inline GatherSmem gather_smem(int D, int S, int ns_used, int mode)
{
    GatherSmem s{};
    const int Sp = (mode == MODE_IID) ? next_pow2(S) : S;
    int off = 0;
    s.O = off; off += (ns_used + 1) * 8;
    s.cr = off; off = (int)align_up((size_t)off + ns_used * 4, 16);
    s.idx = off; off = (int)align_up((size_t)off + Sp * 4, 16);
    s.lead = off; off = (int)align_up((size_t)off + (S + 1) * 4, 16);
    s.acc = off; off += NWARP * D * 4;
    s.misc = off; off += 16 * 4;
    s.total = (int)align_up((size_t)off, 128);
    return s;
}

template <int D>
__global__ void __launch_bounds__(NT) santa_gather_kernel(const Params p)
{
    constexpr int EPL = D / 32;  // V elements per lane
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned FULL = 0xffffffffu;
    const int H_q = p.H_q, G = p.H_q / p.H_kv, L = p.L, S = p.S;
    const int bh = blockIdx.x;
    const int b = bh / H_q, h = bh % H_q, g = h / G;
    int n = p.seq_lens[b];
    if (n < 0 || n > p.n_max) n = 0;  // flagged by the score kernel
    if (n == 0) {
        for (int i = tid; i < D; i += NT) p.out[(size_t)bh * D + i] = 0.f;
        if (p.idx_out)
            for (int i = tid; i < S; i += NT) p.idx_out[(size_t)bh * S + i] = -1;
        return;
    }
    const int ns = (n + L - 1) / L;
    const int ns_used = (p.n_max + L - 1) / L;
    const GatherSmem lay = gather_smem(D, S, ns_used, p.mode);
    double *O = reinterpret_cast<double *>(smem + lay.O);
    int *crs = reinterpret_cast<int *>(smem + lay.cr);
    int *idx = reinterpret_cast<int *>(smem + lay.idx);
    int *lead = reinterpret_cast<int *>(smem + lay.lead);
    float *acc_s = reinterpret_cast<float *>(smem + lay.acc);
    int *misc = reinterpret_cast<int *>(smem + lay.misc);
    const int Sp = (p.mode == MODE_IID) ? next_pow2(S) : S;

    // iid: the S uniforms, sorted (bitonic on the 32-bit draws); independent of the scores
    if (p.mode == MODE_IID) {
        unsigned *uk = reinterpret_cast<unsigned *>(idx);
        for (int s = tid; s < Sp; s += NT) {
            unsigned u = 0xffffffffu;
            if (s < S) {
                uint64_t rnd[4];
                philox_block(p.seed, (uint64_t)(s / 4), b, h, 3, rnd);
                u = (unsigned)(rnd[s % 4] >> 32);
            }
            uk[s] = u;
        }
        __syncthreads();
        for (int kk = 2; kk <= Sp; kk <<= 1)
            for (int jj = kk >> 1; jj > 0; jj >>= 1) {
                for (int s = tid; s < Sp; s += NT) {
                    const int q2 = s ^ jj;
                    if (q2 > s) {
                        const bool asc = (s & kk) == 0;
                        const unsigned x = uk[s], y = uk[q2];
                        if ((x > y) == asc) {
                            uk[s] = y;
                            uk[q2] = x;
                        }
                    }
                }
                __syncthreads();
            }
    }

    pdl_wait();  // the score kernel's results are complete and visible from here on

    // ---- split offsets O_r = sum_{r' < r} W_r' 2^(c_r' - C) (exact scaling, fp64 sums)
    const size_t bhs = (size_t)bh * p.ns_max;
    for (int r = tid; r < ns; r += NT) {
        crs[r] = __ldcg(p.split_c + bhs + r);
        O[r] = __ldcg(p.split_W + bhs + r);
    }
    __syncthreads();
    if (warp == 0) {
        int cm = INT_MIN;
        for (int r = lane; r < ns; r += 32) cm = max(cm, crs[r]);
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) cm = max(cm, __shfl_xor_sync(FULL, cm, m));
        double carry = 0.0;
        for (int base = 0; base < ns; base += 32) {
            const int r = base + lane;
            const double x = r < ns ? __dmul_rn(O[r], pow2d(crs[r] - cm)) : 0.0;
            double incl = x;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double y = __shfl_up_sync(FULL, incl, o);
                if (lane >= o) incl = __dadd_rn(incl, y);
            }
            __syncwarp();
            if (r < ns) O[r] = __dadd_rn(carry, __dsub_rn(incl, x));
            carry = __dadd_rn(carry, __shfl_sync(FULL, incl, 31));
        }
        if (lane == 0) {
            O[ns] = carry;  // Z, in the scale 2^-C
            misc[13] = cm;
        }
    }
    __syncthreads();
    const int Cm = misc[13];
    const double Z = O[ns];

    // ---- points -> split (smem) -> chunk (coff) -> key (w).  Lanes whose points share a
    // split load its chunk offsets once (one line); lanes sharing a chunk load its 32
    // weights once; each lane then binary-searches the shuffled values.
    const size_t bhc = (size_t)bh * p.nch;
    const float *wrow = p.w + (size_t)bh * p.n_pad;
    for (int base = warp * 32; base < S; base += NT) {
        const int s = base + lane;
        const bool act = s < S;
        int rr = 0;
        double Tl = 0.0;
        if (act) {
            double t;
            if (p.mode != MODE_IID) {
                t = sample_point(p.mode, p.seed, b, h, s, p.rS);
            } else {
                t = __dmul_rn(__uint2double_rn(reinterpret_cast<const unsigned *>(idx)[s]), 0x1p-32);
            }
            const double T = __dmul_rn(t, Z);
            const uint64_t Tk = dkey(T);
            int lo = 0, hi = ns - 1;  // largest r with O_r <= T
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (dkey(O[mid]) <= Tk) lo = mid; else hi = mid - 1;
            }
            rr = lo;
            Tl = __dmul_rn(__dsub_rn(T, O[rr]), pow2pos(Cm - crs[rr]));
        }
        int chunk = 0;
        double cbase = 0.0;
        unsigned todo = __ballot_sync(FULL, act);
        while (todo) {
            const int ld = __ffs(todo) - 1;
            const int rL = __shfl_sync(FULL, rr, ld);
            const unsigned gm = __ballot_sync(FULL, act && rr == rL) & todo;
            const int ncr = (min(L, n - rL * L) + CHUNK - 1) / CHUNK;
            const double cl = lane < ncr ? __ldcg(p.coff + bhc + (size_t)rL * (L / CHUNK) + lane) : 0.0;
            const uint64_t Tlk = dkey(Tl);
            int c = 0;
#pragma unroll
            for (int step = 16; step >= 1; step >>= 1) {
                const int cand = c + step;
                const double v = __shfl_sync(FULL, cl, cand & 31);
                if (cand < ncr && dkey(v) <= Tlk) c = cand;
            }
            const double cv = __shfl_sync(FULL, cl, c);
            if ((gm >> lane) & 1u) {
                chunk = c;
                cbase = cv;
            }
            todo &= ~gm;
        }
        int pick = 0;
        todo = __ballot_sync(FULL, act);
        while (todo) {
            const int ld = __ffs(todo) - 1;
            const int rL = __shfl_sync(FULL, rr, ld), cL = __shfl_sync(FULL, chunk, ld);
            const unsigned gm = __ballot_sync(FULL, act && rr == rL && chunk == cL) & todo;
            const int j0 = rL * L + cL * CHUNK;
            const int jn = min(CHUNK, n - j0);
            const float wv = lane < jn ? __ldcg(wrow + j0 + lane) : 0.f;
            const int shift = __ldcg(p.cshift + bhc + (size_t)rL * (L / CHUNK) + cL);
            float P = wv;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(FULL, P, o);
                if (lane >= o) P = __fadd_rn(P, y);
            }
            const unsigned posm = __ballot_sync(FULL, wv > 0.f);
            const int lastpos = posm ? 31 - __clz(posm) : 0;
            // remainder inside the chunk, in the chunk's own scale 2^-c_t
            const float rres = (float)__dmul_rn(__dsub_rn(Tl, cbase), pow2pos(shift));
            int c = -1;  // largest j with P_j <= rres
#pragma unroll
            for (int step = 16; step >= 1; step >>= 1) {
                const int cand = c + step;
                const float v = __shfl_sync(FULL, P, cand < 0 ? 0 : (cand & 31));
                if (cand < 32 && v <= rres) c = cand;
            }
            int jj = c + 1;
            if (jj >= jn) jj = lastpos;  // only when rounding put t past the chunk's mass
            if ((gm >> lane) & 1u) pick = j0 + jj;
            todo &= ~gm;
        }
        if (act) idx[s] = pick;  // (iid: overwrites this point's own uniform)
    }
    __syncthreads();

    // ---- sorted indices out; distinct rows (run starts) and their counts
    if (p.idx_out)
        for (int s = tid; s < S; s += NT) p.idx_out[(size_t)bh * S + s] = idx[s];
    {
        const int per = (S + NT - 1) / NT;
        const int s0 = min(tid * per, S), s1 = min(s0 + per, S);
        int cnt = 0;
        for (int s = s0; s < s1; ++s) cnt += (s == 0 || idx[s] != idx[s - 1]) ? 1 : 0;
        int nlead;
        int pos = block_excl_scan(cnt, misc, &nlead);
        for (int s = s0; s < s1; ++s)
            if (s == 0 || idx[s] != idx[s - 1]) lead[pos++] = s;
        if (tid == 0) lead[nlead] = S;
        __syncthreads();
        // gather-add: warp-strided over the distinct rows, 8 rows in flight per warp
        float acc[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
        const uint16_t *vg = p.v + ((size_t)b * p.H_kv + g) * (size_t)p.n_max * D;
        constexpr int U = 8;
        for (int l0 = warp * U; l0 < nlead; l0 += NWARP * U) {
            float vv[U][EPL];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int li = l0 + u;
                const int j = li < nlead ? idx[lead[li]] : 0;
                if constexpr (EPL == 4) {
                    const uint2 raw = *reinterpret_cast<const uint2 *>(vg + (size_t)j * D + 4 * lane);
                    vv[u][0] = bf16lo_to_f32(raw.x);
                    vv[u][1] = bf16hi_to_f32(raw.x);
                    vv[u][2] = bf16lo_to_f32(raw.y);
                    vv[u][3] = bf16hi_to_f32(raw.y);
                } else {
                    const uint32_t raw = *reinterpret_cast<const uint32_t *>(vg + (size_t)j * D + 2 * lane);
                    vv[u][0] = bf16lo_to_f32(raw);
                    vv[u][1] = bf16hi_to_f32(raw);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int li = l0 + u;
                if (li < nlead) {
                    const float cf = (float)(lead[li + 1] - lead[li]);
#pragma unroll
                    for (int e = 0; e < EPL; ++e) acc[e] = __fmaf_rn(cf, vv[u][e], acc[e]);
                }
            }
        }
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc_s[warp * D + EPL * lane + e] = acc[e];
        __syncthreads();
        for (int i = tid; i < D; i += NT) {
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < NWARP; ++w) sum = __fadd_rn(sum, acc_s[w * D + i]);
            p.out[(size_t)bh * D + i] = __fdiv_rn(sum, (float)S);
        }
    }
}

}  // namespace santa
