// santa_gather.cuh -- SANTA value stage: sample points, CDF search, gather-add, sm_103a.
//
// "Stochastic Sparse Attention for Memory-Bound Inference" (abstract): sample S << n_k
// indices from the post-softmax distribution and aggregate only those value rows,
// scaled by 1/S.  One CTA per (batch row b, query head h), launched as a programmatic
// dependent of the score kernel (its point generation overlaps the score kernel's
// tail).  It
//   1. draws the S sorted points t_s (systematic, stratified, or sorted iid);
//   2. re-scores error-free the keys within tau2 (log2 units) of the head's global
//      maximum score -- found through the split and chunk maxima the score kernel
//      left -- and patches their weights, the chunk offsets after them and the split
//      totals (the heaviest keys' fp32 dot-product rounding would otherwise shift every
//      later CDF boundary);
//   3. merges the split totals exactly: O_r = sum_{r'<r} W_r' 2^(c_r' - C), Z = O_ns;
//   4. maps each point to i_s = min{ j : W_j > t_s Z } by a split -> chunk -> key
//      search, one thread per point with independent loads;
//   5. gather-adds each distinct sampled V row once, weighted by its count, and
//      writes out = sum / S and the sorted indices.
#pragma once

#include "santa_sample.cuh"

namespace santa {

struct GatherSmem {
    int t, O, cr, sm, hot, idx, lead, acc, qf, misc, total;
};

__host__ __device__ inline GatherSmem gather_smem(int D, int S, int ns_used, int mode)
{
    GatherSmem s{};
    const int Sp = (mode == MODE_IID) ? next_pow2(S) : S;
    int off = 0;
    s.t = off; off += S * 8;
    s.O = off; off += (ns_used + 1) * 8;
    s.cr = off; off = (int)align_up((size_t)off + ns_used * 4, 16);
    s.sm = off; off = (int)align_up((size_t)off + ns_used * 4, 16);
    s.hot = off; off = (int)align_up((size_t)off + ns_used * 4, 16);
    s.idx = off; off = (int)align_up((size_t)off + Sp * 4, 16);
    s.lead = off; off = (int)align_up((size_t)off + (S + 1) * 4, 16);
    s.acc = off; off += NWARP * D * 4;
    s.qf = off; off += D * 4;
    s.misc = off; off += 16 * 4;
    s.total = (int)align_up((size_t)off, 128);
    return s;
}

enum : int { GM_CMAX = 13, GM_NHOT = 14, GM_MAX = 15 };

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
    const int cps = L / CHUNK;  // chunks per full split
    const GatherSmem lay = gather_smem(D, S, ns_used, p.mode);
    double *tpt = reinterpret_cast<double *>(smem + lay.t);
    double *O = reinterpret_cast<double *>(smem + lay.O);
    int *crs = reinterpret_cast<int *>(smem + lay.cr);
    float *smx = reinterpret_cast<float *>(smem + lay.sm);
    int *hot = reinterpret_cast<int *>(smem + lay.hot);
    int *idx = reinterpret_cast<int *>(smem + lay.idx);
    int *lead = reinterpret_cast<int *>(smem + lay.lead);
    float *acc_s = reinterpret_cast<float *>(smem + lay.acc);
    float *qf = reinterpret_cast<float *>(smem + lay.qf);
    int *misc = reinterpret_cast<int *>(smem + lay.misc);
    const int Sp = (p.mode == MODE_IID) ? next_pow2(S) : S;

    // ---- 1. points (independent of the scores) and the query head in fp32
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
        for (int s = tid; s < S; s += NT) tpt[s] = __dmul_rn(__uint2double_rn(uk[s]), 0x1p-32);
    } else {
        for (int s = tid; s < S; s += NT) tpt[s] = sample_point(p.mode, p.seed, b, h, s, p.rS);
    }
    for (int i = tid; i < D; i += NT) qf[i] = __uint_as_float((uint32_t)p.q[(size_t)bh * D + i] << 16);
    if (tid == 0) {
        misc[GM_NHOT] = 0;
        misc[GM_MAX] = INT_MIN;  // below the key of every fp32 value
    }

    pdl_wait();  // the score kernel's results are complete and visible from here on

    // ---- 2. split data; the head's maximum score
    const size_t bhs = (size_t)bh * p.ns_max;
    __syncthreads();
    float mloc = __int_as_float(0xff800000);
    for (int r = tid; r < ns; r += NT) {
        crs[r] = __ldcg(p.split_c + bhs + r);
        O[r] = __ldcg(p.split_W + bhs + r);
        smx[r] = __ldcg(p.split_m + bhs + r);
        mloc = fmaxf(mloc, smx[r]);
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(FULL, mloc, m));
    if (lane == 0) atomicMax(misc + GM_MAX, fkey(mloc));
    __syncthreads();
    const float M = fkey_inv(misc[GM_MAX]);
    const float thr = M - p.tau2;
    for (int r = tid; r < ns; r += NT)
        if (smx[r] >= thr) hot[atomicAdd(misc + GM_NHOT, 1)] = r;
    __syncthreads();

    // ---- 3. re-score the keys within tau2 of the maximum; patch w, coff, W_r
    const int nhot = misc[GM_NHOT];
    const size_t bhc = (size_t)bh * p.nch;
    float *wrow = p.w + (size_t)bh * p.n_pad;
    const uint16_t *kg = p.k + ((size_t)b * p.H_kv + g) * (size_t)p.n_max * D;
    for (int hi = warp; hi < nhot; hi += NWARP) {
        const int r = hot[hi];
        const int nck = (min(L, n - r * L) + CHUNK - 1) / CHUNK;
        const size_t cbase = bhc + (size_t)r * cps;
        const bool cact = lane < nck;
        const float cm = cact ? __ldcg(p.cmax + cbase + lane) : __int_as_float(0xff800000);
        const int csh = cact ? __ldcg(p.cshift + cbase + lane) : 0;
        unsigned hm = __ballot_sync(FULL, cact && cm >= thr);
        const int cr = crs[r];
        double dlane = 0.0, dtot = 0.0;
        while (hm) {
            const int c = __ffs(hm) - 1;
            hm &= hm - 1;
            const int ct = cr - __shfl_sync(FULL, csh, c);
            const int j0 = r * L + c * CHUNK;
            const int jn = min(CHUNK, n - j0);
            const float wv = lane < jn ? __ldcg(wrow + j0 + lane) : 0.f;
            const float wthr = exp2f(thr - (float)ct);
            unsigned heavy = __ballot_sync(FULL, lane < jn && wv >= wthr);
            double dch = 0.0;
            while (heavy) {
                const int k = __ffs(heavy) - 1;
                heavy &= heavy - 1;
                float shi, slo;
                refine_score<D>(reinterpret_cast<const uint8_t *>(kg + (size_t)(j0 + k) * D), qf, lane, p.k2_hi,
                                p.k2_lo, shi, slo);
                const float wnew = exp2f(__fadd_rn(__fsub_rn(shi, (float)ct), slo));
                const float wold = __shfl_sync(FULL, wv, k);
                if (lane == 0) wrow[j0 + k] = wnew;
                dch = __dadd_rn(dch, __dsub_rn((double)wnew, (double)wold));
            }
            const double dsp = __dmul_rn(dch, pow2d(ct - cr));
            if (lane > c) dlane = __dadd_rn(dlane, dsp);
            dtot = __dadd_rn(dtot, dsp);
        }
        if (lane < nck && dlane != 0.0) p.coff[cbase + lane] = __dadd_rn(__ldcg(p.coff + cbase + lane), dlane);
        if (lane == 0) O[r] = __dadd_rn(O[r], dtot);
    }
    __syncthreads();

    // ---- 4. split offsets O_r = sum_{r' < r} W_r' 2^(c_r' - C) (exact scaling, fp64 sums)
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
            misc[GM_CMAX] = cm;
        }
    }
    __syncthreads();
    const int Cm = misc[GM_CMAX];
    const double Z = O[ns];

    // ---- 5. points -> split (smem) -> chunk (coff, one line) -> key (w, one line)
    for (int s = tid; s < S; s += NT) {
        const double T = __dmul_rn(tpt[s], Z);
        const uint64_t Tk = dkey(T);
        int lo = 0, hi = ns - 1;  // largest r with O_r <= T
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (dkey(O[mid]) <= Tk) lo = mid; else hi = mid - 1;
        }
        const int r = lo;
        const double Tl = __dmul_rn(__dsub_rn(T, O[r]), pow2pos(Cm - crs[r]));
        const uint64_t Tlk = dkey(Tl);
        const int nck = (min(L, n - r * L) + CHUNK - 1) / CHUNK;
        const size_t cbase = bhc + (size_t)r * cps;
        int cst = 0;
        double cb = 0.0;
#pragma unroll
        for (int c = 1; c < CPS_MAX; ++c) {  // coff of chunk 0 is 0
            if (c < nck) {
                const double v = __ldcg(p.coff + cbase + c);
                if (dkey(v) <= Tlk) {
                    cst = c;
                    cb = v;
                }
            }
        }
        const int shift = __ldcg(p.cshift + cbase + cst);
        const float rres = (float)__dmul_rn(__dsub_rn(Tl, cb), pow2pos(shift));
        const int j0 = r * L + cst * CHUNK;
        const int jn = min(CHUNK, n - j0);
        const float4 *w4 = reinterpret_cast<const float4 *>(wrow + j0);
        float wv[CHUNK];
#pragma unroll
        for (int k4 = 0; k4 < CHUNK / 4; ++k4) {
            const float4 x = __ldcg(w4 + k4);
            wv[4 * k4] = x.x;
            wv[4 * k4 + 1] = x.y;
            wv[4 * k4 + 2] = x.z;
            wv[4 * k4 + 3] = x.w;
        }
        float P = 0.f;
        int pick = -1, lastpos = 0;
#pragma unroll
        for (int k = 0; k < CHUNK; ++k) {
            const float x = k < jn ? wv[k] : 0.f;
            P = __fadd_rn(P, x);
            if (x > 0.f) lastpos = k;
            if (pick < 0 && P > rres) pick = k;
        }
        if (pick < 0) pick = lastpos;  // only when rounding put t past the chunk's mass
        idx[s] = j0 + pick;            // (iid: overwrites this point's own uniform)
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
