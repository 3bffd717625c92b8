// santa_score.cuh -- SANTA score stage: scores, weights and the CDF pieces, sm_103a.
//
// "Stochastic Sparse Attention for Memory-Bound Inference" (abstract): the score stage
// reads all n_k cached keys and forms the post-softmax distribution from which the
// value stage samples.  This persistent kernel streams every split (b, g, r) -- L keys
// of KV head g of batch row b -- once, as 16 KB tiles through an NSTAGE-deep ring of
// 1-D TMA bulk copies, and leaves in the workspace, per query head of the group:
//   w_j      fp32 weight 2^(s_j log2 e - c_t) of every key (c_t: the integer scale of
//            the key's tile, >= the running maximum, so w_j <= 1)
//   coff     fp64 exclusive prefix of the 32-key chunk totals within the split, in the
//            split's scale 2^-c_r, and cshift = c_r - c_t of each chunk
//   split_W  fp64 split total and split_c = c_r (the integer scale of the split)
// Chunk totals are exact (64-bit fixed-point sums of the fp32 weights); rescaling is by
// powers of two, so the CDF that the value stage assembles from these pieces has no
// rounding beyond that of the fp32 weights themselves.
//
// Scores within tau2 (log2 units) of the running maximum are recomputed error-free
// (double-float dot product of the staged row), because the heaviest keys' rounding
// errors would otherwise shift every later CDF boundary.
//
// Per tile the CTA synchronises once: after the wait for the tile's data.  The weights
// and chunk totals of a tile are computed in the iteration after its scores (its
// scores and the CTA-wide maxima are then visible), and a split's chunk prefix one
// iteration later still; the last tile's work is drained after the loop.
#pragma once

#include "santa_sample.cuh"

namespace santa {

struct ScoreSmem {
    int stage, bar, desc, qf, tmax, misc, nb, prefix, sc, chk_tot, chk_exp, total;
};

__host__ __device__ inline ScoreSmem score_smem(int D, int G, int B, int nstage)
{
    const int TK = (D == 128) ? 64 : 128;
    ScoreSmem s{};
    int off = 0;
    s.stage = off; off += nstage * TILE_BYTES;
    s.bar = off; off += nstage * 8;
    s.desc = off; off = (int)align_up((size_t)off + nstage * 16, 16);
    s.qf = off; off += G * D * 4;
    s.tmax = off; off += G * NWARP * 4;
    s.misc = off; off += 16 * 4;
    s.nb = off; off += (int)align_up((size_t)B * 4, 16);
    s.prefix = off; off += (int)align_up((size_t)(B + 1) * 4, 16);
    off = (int)align_up((size_t)off, 16);
    s.sc = off; off += 2 * 2 * G * TK * 4;
    off = (int)align_up((size_t)off, 16);
    s.chk_tot = off; off += 2 * G * (LMAX / CHUNK) * 8;
    s.chk_exp = off; off += 2 * G * (LMAX / CHUNK) * 4;
    s.total = (int)align_up((size_t)off, 128);
    return s;
}

template <int D, int G, int NSTAGE>
__global__ void __launch_bounds__(NT, (G <= 4 ? 2 : 1)) santa_score_kernel(const Params p)
{
    using C = SampleCfg<D, G>;
    constexpr int TK = C::TK;
    constexpr int CPT = TK / CHUNK;    // chunks per tile
    constexpr int NCH = LMAX / CHUNK;  // chunks per split, at most
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sub = lane % C::P, grp = lane / C::P;
    const int B = p.B, H_kv = p.H_kv, H_q = p.H_q, L = p.L;
    const ScoreSmem lay = score_smem(D, G, B, NSTAGE);

    uint8_t *stage = smem + lay.stage;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + lay.bar);
    int4 *sdesc = reinterpret_cast<int4 *>(smem + lay.desc);
    float *qf = reinterpret_cast<float *>(smem + lay.qf);
    float *tmax = reinterpret_cast<float *>(smem + lay.tmax);
    int *misc = reinterpret_cast<int *>(smem + lay.misc);
    int *nb = reinterpret_cast<int *>(smem + lay.nb);
    int *prefix = reinterpret_cast<int *>(smem + lay.prefix);
    float *scb = reinterpret_cast<float *>(smem + lay.sc);  // [buf][hi|lo][G][TK]
    long long *chk_tot = reinterpret_cast<long long *>(smem + lay.chk_tot);  // [parity][G][NCH]
    int *chk_exp = reinterpret_cast<int *>(smem + lay.chk_exp);        // [parity][G][NCH]
    const float NEG_INF = __int_as_float(0xff800000);

    build_item_space(p, nb, prefix, misc);
    if (tid == 0) {
        for (int s = 0; s < NSTAGE; ++s) mbar_init(&bars[s], 1);
        mbar_fence_init();
    }
    __syncthreads();
    const int total_items = prefix[B];

    // ---- producer (thread 0): the tiles of the items it takes, in order
    int pr_item = 0, pr_tile = 0, pr_ntiles = 0, pr_valid = 0, pr_next = 0;
    long long pr_row0 = 0;
    bool pr_end = false;
    uint64_t policy = 0;
    if (tid == 0) {
        policy = l2_policy_evict_first();
        pr_next = atomicAdd(p.ctrl + CTRL_WORK, 1);
    }
    auto produce = [&](int slot) {
        while (!pr_end && pr_tile == pr_ntiles) {
            const int it = pr_next;
            if (it < 0 || it >= total_items) {
                pr_end = true;
                break;
            }
            pr_next = atomicAdd(p.ctrl + CTRL_WORK, 1);
            const Item x = decode_item(it, prefix, nb, B, H_kv, L);
            if (x.n == 0) continue;  // empty rows are written by the value stage
            pr_item = it;
            pr_tile = 0;
            pr_valid = min(L, x.n - x.r * L);
            pr_ntiles = (pr_valid + TK - 1) / TK;
            pr_row0 = ((long long)x.b * H_kv + x.g) * p.n_max + (long long)x.r * L;
        }
        if (pr_end) {
            sdesc[slot] = make_int4(DESC_END, 0, 0, 0);
            mbar_arrive(&bars[slot]);
            return;
        }
        const int rows = min(TK, pr_valid - pr_tile * TK);
        const int flags = (pr_tile == pr_ntiles - 1) ? FLAG_LAST : 0;
        sdesc[slot] = make_int4(pr_item, pr_tile, rows, flags);
        const uint32_t bytes = (uint32_t)rows * C::ROWB;
        mbar_arrive_tx(&bars[slot], bytes);
        bulk_g2s(stage + slot * TILE_BYTES, p.k + (pr_row0 + (long long)pr_tile * TK) * D, bytes, &bars[slot],
                 policy);
        ++pr_tile;
    };
    if (tid == 0)
        for (int s = 0; s < NSTAGE; ++s) produce(s);

    // ---- consumer state (uniform across the CTA)
    unsigned long long qp[G][8];
    float runmax[G];
#pragma unroll
    for (int h = 0; h < G; ++h) runmax[h] = NEG_INF;
    Item cur{0, 0, 0, 0, 1};
    int parity = 0;  // chunk buffer of the current split
    // pending tile (weights not yet written) and pending split (prefix not yet written)
    bool pt_ok = false, pt_last = false;
    int pt_buf = 0, pt_rows = 0, pt_tile = 0, pt_par = 0, pt_valid = 0;
    Item pt_item{0, 0, 0, 0, 1};
    bool fz_ok = false;
    int fz_par = 0, fz_valid = 0;
    Item fz_item{0, 0, 0, 0, 1};
    bool aborted = false;
    int it = 0;

    // weights and exact chunk totals of the pending tile: one key per thread, a warp per
    // 32-key chunk; the chunk total is an exact sum in 64-bit fixed point (2^-50 units of
    // the chunk's scale 2^c_t; every weight is at most ~1, so 32 of them fit easily)
    auto tile_weights = [&]() {
        const float *hi_b = scb + pt_buf * 2 * G * TK;
        const float *lo_b = hi_b + G * TK;
        const size_t bh0 = (size_t)pt_item.b * H_q + (size_t)pt_item.g * G;
        for (int e0 = warp * 32; e0 < G * TK; e0 += NT) {  // whole warps (they shuffle)
            const int e = e0 + lane;
            const int h = e / TK, key = e % TK;
            float rm = runmax[0];
#pragma unroll
            for (int hh = 1; hh < G; ++hh) rm = (h == hh) ? runmax[hh] : rm;
            const int ct = (int)ceilf(fminf(fmaxf(rm, -16777216.f), 16777216.f));
            float w = 0.f;
            if (key < pt_rows) {
                w = exp2f(__fadd_rn(__fsub_rn(hi_b[h * TK + key], (float)ct), lo_b[h * TK + key]));
                p.w[(bh0 + h) * p.n_pad + (size_t)pt_item.r * L + (size_t)pt_tile * TK + key] = w;
            }
            long long v = fixed50(w);
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
            if (lane == 0) {
                const int k = pt_tile * CPT + key / CHUNK;
                chk_tot[(pt_par * G + h) * NCH + k] = v;
                chk_exp[(pt_par * G + h) * NCH + k] = ct;
            }
        }
    };
    // chunk prefix, split total and scales of the pending split (warp h for head h)
    auto split_finalize = [&]() {
        const int nchunks = (fz_valid + CHUNK - 1) / CHUNK;
        if (warp < G) {
            const int h = warp;
            const size_t bh = (size_t)fz_item.b * H_q + (size_t)fz_item.g * G + h;
            double tot = 0.0;
            int ce = INT_MIN;
            if (lane < nchunks) {
                tot = __dmul_rn(__ll2double_rn(chk_tot[(fz_par * G + h) * NCH + lane]), 0x1p-50);
                ce = chk_exp[(fz_par * G + h) * NCH + lane];
            }
            int cr = ce;
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) cr = max(cr, __shfl_xor_sync(0xffffffffu, cr, m));
            const double x = lane < nchunks ? __dmul_rn(tot, pow2d(ce - cr)) : 0.0;
            double incl = x;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl = __dadd_rn(incl, y);
            }
            if (lane < nchunks) {
                const size_t ci = bh * p.nch + (size_t)fz_item.r * (L / CHUNK) + lane;
                p.coff[ci] = __dsub_rn(incl, x);
                p.cshift[ci] = cr - ce;
            }
            const double W = __shfl_sync(0xffffffffu, incl, 31);
            if (lane == 0) {
                p.split_W[bh * p.ns_max + fz_item.r] = W;
                p.split_c[bh * p.ns_max + fz_item.r] = cr;
            }
        }
    };
    auto fold_tmax = [&]() {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float4 a = *reinterpret_cast<const float4 *>(tmax + h * NWARP);
            const float4 c = *reinterpret_cast<const float4 *>(tmax + h * NWARP + 4);
            runmax[h] = fmaxf(runmax[h], fmaxf(fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w)),
                                               fmaxf(fmaxf(c.x, c.y), fmaxf(c.z, c.w))));
        }
    };
    auto retire_pending = [&]() {
        if (fz_ok) {
            split_finalize();
            fz_ok = false;
        }
        if (pt_ok) {
            tile_weights();
            if (pt_last) {
                fz_ok = true;
                fz_item = pt_item;
                fz_par = pt_par;
                fz_valid = pt_valid;
            }
            pt_ok = false;
        }
    };

    for (;; ++it) {
        const int slot = it % NSTAGE;
        const uint32_t par = (uint32_t)(it / NSTAGE) & 1u;
        const bool ok = mbar_wait_bounded(&bars[slot], par, p.wait_ns);
        if (__syncthreads_or(!ok)) {
            aborted = true;
            break;
        }
        // everyone is done with the previous tile: refill its slot, fold its maxima in,
        // and retire the work that was waiting for this barrier
        if (tid == 0 && it > 0) produce((it - 1) % NSTAGE);
        if (pt_ok) fold_tmax();
        retire_pending();
        const int4 dsc = sdesc[slot];
        if (dsc.x == DESC_END) break;

        const int tile = dsc.y, rows = dsc.z;
        if (tile == 0) {
            cur = decode_item(dsc.x, prefix, nb, B, H_kv, L);
            parity ^= 1;
            const uint16_t *qg = p.q + ((size_t)cur.b * H_q + (size_t)cur.g * G) * D;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const uint4 a = *reinterpret_cast<const uint4 *>(qg + h * D + 8 * sub);
                const uint4 c = *reinterpret_cast<const uint4 *>(qg + h * D + 8 * (sub + C::P));
                const uint32_t wv[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) qp[h][i] = bf16x2_to_f32x2(wv[i]);
                runmax[h] = NEG_INF;
            }
            for (int i = tid; i < G * D / 2; i += NT) {
                const uint32_t w2 = *reinterpret_cast<const uint32_t *>(qg + 2 * i);
                qf[2 * i] = bf16lo_to_f32(w2);
                qf[2 * i + 1] = bf16hi_to_f32(w2);
            }
            __syncthreads();
        }

        // ---- scores of this tile: warp `warp` takes keys [warp*KW, warp*KW + KW)
        const int buf = it & 1;
        float *sc_hi = scb + buf * 2 * G * TK;
        float *sc_lo = sc_hi + G * TK;
        const uint8_t *tb = stage + slot * TILE_BYTES;
        const int kwarp = warp * C::KW;
        const int kbase = kwarp + 2 * grp;
        float val[2 * G];
        tile_dots<D, G>(tb, kbase, sub, qp, val);
        float s2[C::NV];
        bool own[C::NV];
#pragma unroll
        for (int i = 0; i < C::NV; ++i) {
            const int key = kbase + C::key2_of(lane, i);
            own[i] = (sub % C::REP) == 0 && key < rows;
            s2[i] = key < rows ? __fmul_rn(val[i], p.k2_hi) : NEG_INF;
            if ((sub % C::REP) == 0) {
                const int h = C::head_of(lane, i);
                sc_hi[h * TK + key] = s2[i];
                sc_lo[h * TK + key] = 0.f;
            }
        }
        float wm[C::NV];
#pragma unroll
        for (int i = 0; i < C::NV; ++i) wm[i] = s2[i];
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            if (C::SAME & (unsigned)m) {
#pragma unroll
                for (int i = 0; i < C::NV; ++i) wm[i] = fmaxf(wm[i], __shfl_xor_sync(0xffffffffu, wm[i], m));
            }
        }
        if ((lane & C::SAME) == 0) {
#pragma unroll
            for (int i = 0; i < C::NV; ++i) tmax[C::head_of(lane, i) * NWARP + warp] = wm[i];
        }
        if (tile == 0) {
            // first tile of a split: base the window on the whole tile's maximum
            __syncthreads();
            fold_tmax();
        }
        // recompute, error-free, the scores within tau2 of the split's running maximum
#pragma unroll
        for (int i = 0; i < C::NV; ++i) {
            const int h = C::head_of(lane, i);
            float rm = runmax[0];
#pragma unroll
            for (int hh = 1; hh < G; ++hh) rm = (h == hh) ? runmax[hh] : rm;
            const float thr = fmaxf(rm, wm[i]) - p.tau2;
            unsigned cand = __ballot_sync(0xffffffffu, own[i] && s2[i] >= thr);
            while (cand) {
                const int src = __ffs(cand) - 1;
                cand &= cand - 1;
                const int key = kwarp + 2 * (src / C::P) + C::key2_of(src, i);
                const int hh = C::head_of(src, i);
                float hi, lo;
                refine_score<D>(tb + key * C::ROWB, qf + hh * D, lane, p.k2_hi, p.k2_lo, hi, lo);
                if (lane == 0) {
                    sc_hi[hh * TK + key] = hi;
                    sc_lo[hh * TK + key] = lo;
                }
            }
        }
        // this tile's weights are written next iteration (after the barrier)
        pt_ok = true;
        pt_last = (dsc.w & FLAG_LAST) != 0;
        pt_buf = buf;
        pt_rows = rows;
        pt_tile = tile;
        pt_par = parity;
        pt_item = cur;
        pt_valid = min(L, cur.n - cur.r * L);
    }

    if (!aborted) {
        // drain: the last tile's weights, then the last split's prefix
        __syncthreads();
        if (pt_ok) fold_tmax();
        retire_pending();
        __syncthreads();
        retire_pending();
    } else {
        // give the copies still in flight a bounded chance to land before the CTA exits
        if (tid == 0) {
            set_dev_error(p.ctrl, DEV_TIMEOUT);
            for (int k = 0; k < NSTAGE - 1; ++k) {
                const int j = it + k;
                mbar_wait_bounded(&bars[j % NSTAGE], (uint32_t)(j / NSTAGE) & 1u, p.wait_ns);
            }
        }
        __syncthreads();
    }
    __threadfence();
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
