// santa_score.cuh -- SANTA score stage: scores, weights and the CDF pieces, sm_103a.
//
// "Stochastic Sparse Attention for Memory-Bound Inference" (abstract): the score stage
// reads all n_k cached keys and forms the post-softmax distribution from which the
// value stage samples.  This is the kernel that streams the K cache (about 97% of the
// bytes of a sampled decode step), so it is built for bandwidth:
//
//  * persistent CTAs of 8 independent warps; a warp takes a whole split (b, g, r) --
//    L consecutive keys of KV head g of batch row b -- from a global work counter and
//    streams it through its own ring of 32-key tiles, filled by 1-D TMA bulk copies
//    (cp.async.bulk, completion on an mbarrier) that lane 0 issues;
//  * no CTA-wide barrier after the prologue: a warp waits only for its own tiles;
//  * one 32-key tile is one CDF chunk, so every per-chunk quantity is a warp-local
//    reduction over the lanes that hold the same query head.
//
// Per query head of the group it leaves in the workspace:
//   w_j      fp32 weight 2^(s_j log2 e - c_t), c_t = ceil of the split's running maximum
//            (in log2 units) at the key's chunk, so w_j <= 1
//   cmax     the chunk's maximum of s_j log2 e (fp32)
//   coff     fp64 exclusive prefix of the chunk totals within the split, in the split's
//            scale 2^-c_r, and cshift = c_r - c_t of each chunk
//   split_W  fp64 split total, split_c = c_r, split_m = the split's maximum score
// Rescaling between chunk and split scales is by powers of two (exact in fp64).
//
// Weights are computed with one rounding of the small exponent s log2e - c_t (two
// fused multiply-adds with scale*log2e split into an fp32 pair), so the keys at the
// top of the distribution carry only the dot product's own rounding.  The value stage
// later re-scores error-free the few keys within tau2 of the global maximum (found
// from cmax), where that rounding would move later CDF boundaries most.
#pragma once

#include "santa_sample.cuh"

namespace santa {

template <int D>
struct ScoreTile {
    static constexpr int KEYS = CHUNK;                 // keys per warp tile = one CDF chunk
    static constexpr int BYTES = KEYS * 2 * D;         // 8 KB at d=128, 4 KB at d=64
    static constexpr int NSTAGE = 24576 / BYTES;       // 24 KB of ring per warp
};

struct ScoreSmem {
    int nb, prefix, misc, warp0, warp_bytes, ring, bar, desc, ctot, cexp, total;
};

__host__ __device__ inline ScoreSmem score_smem(int D, int G, int B)
{
    const int bytes = CHUNK * 2 * D;
    const int nstage = 24576 / bytes;
    ScoreSmem s{};
    int off = 0;
    s.nb = off; off += (int)align_up((size_t)B * 4, 16);
    s.prefix = off; off += (int)align_up((size_t)(B + 1) * 4, 16);
    s.misc = off; off += 16 * 4;
    s.warp0 = (int)align_up((size_t)off, 128);
    // per-warp block (offsets relative to the warp's base)
    int w = 0;
    s.ring = w; w += nstage * bytes;
    s.bar = w; w += nstage * 8;
    s.desc = w = (int)align_up((size_t)w, 16); w += nstage * 16;
    s.ctot = w; w += G * CPS_MAX * 4;
    s.cexp = w; w += G * CPS_MAX * 4;
    s.warp_bytes = (int)align_up((size_t)w, 128);
    s.total = s.warp0 + NWARP * s.warp_bytes;
    return s;
}

template <int D, int G>
__global__ void __launch_bounds__(NT, 1) santa_score_kernel(const Params p)
{
    using C = SampleCfg<D, G>;
    using T = ScoreTile<D>;
    constexpr int NSTAGE = T::NSTAGE;
    constexpr int NCALL = T::KEYS / C::KW;  // tile_dots calls per tile
    constexpr int NV = C::NV;
    constexpr unsigned FULL = 0xffffffffu;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sub = lane % C::P, grp = lane / C::P;
    const int B = p.B, H_kv = p.H_kv, H_q = p.H_q, L = p.L;
    const ScoreSmem lay = score_smem(D, G, B);
    int *nb = reinterpret_cast<int *>(smem + lay.nb);
    int *prefix = reinterpret_cast<int *>(smem + lay.prefix);
    int *misc = reinterpret_cast<int *>(smem + lay.misc);
    uint8_t *wb = smem + lay.warp0 + warp * lay.warp_bytes;
    uint8_t *ring = wb + lay.ring;
    uint64_t *bars = reinterpret_cast<uint64_t *>(wb + lay.bar);
    int4 *desc = reinterpret_cast<int4 *>(wb + lay.desc);
    float *ctot = reinterpret_cast<float *>(wb + lay.ctot);  // [G][CPS_MAX]
    int *cexp = reinterpret_cast<int *>(wb + lay.cexp);      // [G][CPS_MAX]
    const float NEG_INF = __int_as_float(0xff800000);

    build_item_space(p, nb, prefix, misc);
    if (lane == 0) {
        for (int s = 0; s < NSTAGE; ++s) mbar_init(&bars[s], 1);
        mbar_fence_init();
    }
    __syncthreads();  // the only CTA-wide barrier of the main path
    const int total_items = prefix[B];

    // ---- producer state (warp-uniform; lane 0 issues the copies and the atomics)
    uint64_t policy = 0;
    int pend = 0;  // lane 0: the next item index, fetched one item ahead
    if (lane == 0) {
        policy = l2_policy_evict_first();
        pend = atomicAdd(p.ctrl + CTRL_WORK, 1);
    }
    int pr_item = 0, pr_tile = 0, pr_ntiles = 0, pr_valid = 0;
    long long pr_row0 = 0;
    bool pr_end = false;
    auto produce = [&](int slot) {
        while (!pr_end && pr_tile == pr_ntiles) {
            const int it = __shfl_sync(FULL, pend, 0);
            if (it >= total_items) {
                pr_end = true;
                break;
            }
            if (lane == 0) pend = atomicAdd(p.ctrl + CTRL_WORK, 1);
            const Item x = decode_item(it, prefix, nb, B, H_kv, L);
            if (x.n == 0) continue;  // empty rows are written by the value stage
            pr_item = it;
            pr_tile = 0;
            pr_valid = min(L, x.n - x.r * L);
            pr_ntiles = (pr_valid + T::KEYS - 1) / T::KEYS;
            pr_row0 = ((long long)x.b * H_kv + x.g) * p.n_max + (long long)x.r * L;
        }
        if (pr_end) {
            if (lane == 0) desc[slot] = make_int4(DESC_END, 0, 0, 0);
            return;
        }
        const int rows = min(T::KEYS, pr_valid - pr_tile * T::KEYS);
        if (lane == 0) {
            desc[slot] = make_int4(pr_item, pr_tile, rows, pr_tile == pr_ntiles - 1 ? FLAG_LAST : 0);
            const uint32_t bytes = (uint32_t)rows * C::ROWB;
            mbar_arrive_tx(&bars[slot], bytes);
            bulk_g2s(ring + slot * T::BYTES, p.k + (pr_row0 + (long long)pr_tile * T::KEYS) * D, bytes,
                     &bars[slot], policy);
        }
        ++pr_tile;
    };
    for (int s = 0; s < NSTAGE; ++s) produce(s);

    // ---- consumer state (warp-uniform except for the per-lane head slots)
    unsigned long long qp[G][8];
    float runmax[NV];
    Item cur{0, 0, 0, 0, 1};
    bool aborted = false;
    int it = 0;
    for (;; ++it) {
        const int slot = it % NSTAGE;
        __syncwarp();
        const int4 dsc = desc[slot];
        if (dsc.x == DESC_END) break;
        if (!mbar_wait_bounded(&bars[slot], (uint32_t)(it / NSTAGE) & 1u, p.wait_ns)) {
            aborted = true;
            break;
        }
        const int tile = dsc.y, rows = dsc.z;
        if (tile == 0) {
            // a new split: its group's query heads into registers (fp32 pairs of the
            // lane's two 16-byte chunks of each head)
            cur = decode_item(dsc.x, prefix, nb, B, H_kv, L);
            const uint16_t *qg = p.q + ((size_t)cur.b * H_q + (size_t)cur.g * G) * D;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const uint4 a = __ldg(reinterpret_cast<const uint4 *>(qg + h * D + 8 * sub));
                const uint4 c = __ldg(reinterpret_cast<const uint4 *>(qg + h * D + 8 * (sub + C::P)));
                const uint32_t wv[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) qp[h][i] = bf16x2_to_f32x2(wv[i]);
            }
#pragma unroll
            for (int i = 0; i < NV; ++i) runmax[i] = NEG_INF;
        }

        // ---- dot products: call c covers keys [c*KW, c*KW + KW) of the tile
        const uint8_t *tb = ring + slot * T::BYTES;
        float sc[NCALL][NV];
#pragma unroll
        for (int c = 0; c < NCALL; ++c) {
            float val[2 * G];
            tile_dots<D, G>(tb, c * C::KW + 2 * grp, sub, qp, val);
#pragma unroll
            for (int i = 0; i < NV; ++i) sc[c][i] = val[i];
        }
        __syncwarp();
        produce(slot);  // the tile's data is in registers: refill its slot now

        // ---- chunk maximum (log2 units), running maximum and the chunk's scale c_t
        const bool own = (sub % C::REP) == 0;
        float tmx[NV], ct[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            float m = NEG_INF;
#pragma unroll
            for (int c = 0; c < NCALL; ++c) {
                const int key = c * C::KW + 2 * grp + C::key2_of(lane, i);
                if (key < rows) m = fmaxf(m, __fmul_rn(sc[c][i], p.k2_hi));
            }
#pragma unroll
            for (int msk = 1; msk < 32; msk <<= 1)
                if (C::SAME & (unsigned)msk) m = fmaxf(m, __shfl_xor_sync(FULL, m, msk));
            tmx[i] = m;
            runmax[i] = fmaxf(runmax[i], m);
            ct[i] = ceilf(fminf(fmaxf(runmax[i], -16777216.f), 16777216.f));
        }

        // ---- weights (stored), chunk totals
        const size_t bh0 = (size_t)cur.b * H_q + (size_t)cur.g * G;
        const size_t jbase = (size_t)cur.r * L + (size_t)tile * T::KEYS;
        float tot[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int h = C::head_of(lane, i);
            float* wrow = p.w + (bh0 + h) * p.n_pad + jbase;
            float acc = 0.f;
#pragma unroll
            for (int c = 0; c < NCALL; ++c) {
                const int key = c * C::KW + 2 * grp + C::key2_of(lane, i);
                if (key < rows) {
                    const float e = __fmaf_rn(sc[c][i], p.k2_lo, __fmaf_rn(sc[c][i], p.k2_hi, -ct[i]));
                    const float w = exp2f(e);
                    if (own) {
                        wrow[key] = w;
                        acc = __fadd_rn(acc, w);
                    }
                }
            }
#pragma unroll
            for (int msk = 1; msk < 32; msk <<= 1)
                if (C::SAME & (unsigned)msk) acc = __fadd_rn(acc, __shfl_xor_sync(FULL, acc, msk));
            tot[i] = acc;
        }
        // one lane per head records the chunk (lane bits outside SAME select the head)
        const int cidx = tile;  // chunk index within the split
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            if ((lane & C::SAME) == 0 && own) {
                const int h = C::head_of(lane, i);
                ctot[h * CPS_MAX + cidx] = tot[i];
                cexp[h * CPS_MAX + cidx] = (int)ct[i];
                p.cmax[(bh0 + h) * p.nch + (size_t)cur.r * (L / CHUNK) + cidx] = tmx[i];
                if (dsc.w & FLAG_LAST) p.split_m[(bh0 + h) * p.ns_max + cur.r] = runmax[i];
            }
        }

        // ---- split end: chunk prefix within the split, split total and scales.  Lanes
        // form 32/CPS_MAX segments of CPS_MAX lanes, one head per segment and pass.
        if (dsc.w & FLAG_LAST) {
            __syncwarp();
            const int nchunks = tile + 1;
            constexpr int SEG = CPS_MAX, HPP = 32 / SEG;
            const int c = lane % SEG;
#pragma unroll
            for (int h0 = 0; h0 < G; h0 += HPP) {
                const int h = h0 + lane / SEG;
                const bool act = h < G && c < nchunks;
                float x32 = 0.f;
                int ce = INT_MIN;
                if (act) {
                    x32 = ctot[h * CPS_MAX + c];
                    ce = cexp[h * CPS_MAX + c];
                }
                int cr = ce;
#pragma unroll
                for (int msk = SEG / 2; msk >= 1; msk >>= 1) cr = max(cr, __shfl_xor_sync(FULL, cr, msk));
                const double x = act ? __dmul_rn((double)x32, pow2d(ce - cr)) : 0.0;
                double incl = x;
#pragma unroll
                for (int o = 1; o < SEG; o <<= 1) {
                    const double y = __shfl_up_sync(FULL, incl, o);
                    if (c >= o) incl = __dadd_rn(incl, y);
                }
                const size_t bh = bh0 + (size_t)(h < G ? h : 0);
                if (act) {
                    const size_t ci = bh * p.nch + (size_t)cur.r * (L / CHUNK) + c;
                    p.coff[ci] = __dsub_rn(incl, x);
                    p.cshift[ci] = cr - ce;
                }
                if (h < G && c == SEG - 1) {
                    p.split_W[bh * p.ns_max + cur.r] = incl;
                    p.split_c[bh * p.ns_max + cur.r] = cr;
                }
            }
        }
    }

    if (aborted) {
        // give the copies still in flight a bounded chance to land before the CTA exits
        if (lane == 0) {
            set_dev_error(p.ctrl, DEV_TIMEOUT);
            for (int k = 0; k < NSTAGE; ++k) {
                const int j = it + k;
                if (desc[j % NSTAGE].x != DESC_END)
                    mbar_wait_bounded(&bars[j % NSTAGE], (uint32_t)(j / NSTAGE) & 1u, p.wait_ns);
            }
        }
        __syncwarp();
    }
    __threadfence();
    __syncthreads();
    pdl_launch_dependents();
    if (tid == 0) {
        const int done = atomicAdd(p.ctrl + CTRL_EXIT, 1);
        if (done == (int)gridDim.x - 1) {
            p.ctrl[CTRL_WORK] = 0;
            p.ctrl[CTRL_EXIT] = 0;
        }
    }
}

}  // namespace santa
