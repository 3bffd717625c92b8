// santa_score.cuh -- SANTA score stage: scores, weights and per-chunk CDF pieces, sm_103a.
//
// "Stochastic Sparse Attention for Memory-Bound Inference" (abstract): the score stage
// reads all n_k cached keys and forms the post-softmax distribution from which the
// value stage samples.  This is the kernel that streams the K cache (about 97% of the
// bytes of a sampled decode step), so it is built for bandwidth:
//
//  * persistent CTAs of 8 independent warps; a warp takes work units of L consecutive
//    keys of one KV head g of one batch row b -- a static contiguous block of units
//    first, then grabs from a global counter that shrink to single units near the end,
//    so that the warps finish together -- and streams them through its own ring of 32-key tiles, filled by 1-D TMA bulk copies (cp.async.bulk, completion
//    on an mbarrier) that lane 0 issues; K is read with an L2 evict-first hint, and the
//    weights and chunk data are written with evict-last, for the value stage;
//  * the group's query heads ride along with the first tile of a new (b, g) as a second
//    bulk copy on the same barrier, so a warp does not stall on a query load;
//  * no CTA-wide barrier after the prologue: a warp waits only for its own tiles;
//  * one tile is one CDF chunk of 32 keys with its own power-of-two scale, so chunks
//    are independent: nothing is carried from one tile to the next.
//
// Per query head of the group and per chunk it leaves in the workspace:
//   w_j    fp32 weight 2^(s_j log2 e - c_t), c_t = ceil(the chunk's maximum of s log2 e),
//          so every w_j <= 1 and the chunk's heaviest key has w > 1/2
//   ctot   the chunk total of the w_j (fp32, summed over the warp in a fixed tree)
//   cexp   c_t (int32)
//   cmax   the chunk's maximum of s log2 e (fp32)
// The value stage turns these into one exact fixed-point prefix per head.
//
// Weights are computed with one rounding of the small exponent s log2e - c_t (two
// fused multiply-adds with scale*log2e split into an fp32 pair), so the keys at the
// top of the distribution carry only the dot product's own rounding.  The value stage
// re-scores error-free the few keys within tau2 of the global maximum (found from
// cmax), where that rounding would move later CDF boundaries most.
#pragma once

#include "santa_sample.cuh"

namespace santa {

template <int D, int G>
struct ScoreTile {
    static constexpr int KEYS = CHUNK;                   // keys per warp tile = one CDF chunk
    static constexpr int BYTES = KEYS * 2 * D;           // 8 KB at d=128, 4 KB at d=64
    static constexpr int NSTAGE = 24576 / BYTES;         // 24 KB of ring per warp
    static constexpr int QBYTES = G * D * 2;             // the group's query heads, bf16
    static constexpr int QBUF = QBYTES <= 1024 ? 2 : 1;  // staging buffers for them
};

struct ScoreSmem {
    int nb, prefix, misc, warp0, warp_bytes, ring, qbuf, bar, desc, total;
};

__host__ __device__ inline ScoreSmem score_smem(int D, int G, int B)
{
    const int bytes = CHUNK * 2 * D;
    const int nstage = 24576 / bytes;
    const int qbytes = G * D * 2;
    const int qbuf = qbytes <= 1024 ? 2 : 1;
    ScoreSmem s{};
    int off = 0;
    s.nb = off; off += (int)align_up((size_t)B * 4, 16);
    s.prefix = off; off += (int)align_up((size_t)(B + 1) * 4, 16);
    s.misc = off; off += 16 * 4;
    s.warp0 = (int)align_up((size_t)off, 128);
    // per-warp block (offsets relative to the warp's base)
    int w = 0;
    s.ring = w; w += nstage * bytes;
    s.qbuf = w; w += qbuf * qbytes;
    s.bar = w; w += nstage * 8;
    s.desc = w = (int)align_up((size_t)w, 16); w += nstage * 16;
    s.warp_bytes = (int)align_up((size_t)w, 128);
    s.total = s.warp0 + NWARP * s.warp_bytes;
    return s;
}


template <int D, int G>
__global__ void __launch_bounds__(NT, 1) santa_score_kernel(const Params p)
{
    using C = SampleCfg<D, G>;
    using T = ScoreTile<D, G>;
    constexpr int NSTAGE = T::NSTAGE;
    constexpr int NCALL = T::KEYS / C::KW;  // tile_dots calls per tile
    constexpr int NV = C::NV;
    constexpr unsigned FULL = 0xffffffffu;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sub = lane % C::P, grp = lane / C::P;
    const int B = p.B, H_kv = p.H_kv, L = p.L;  // L: keys per work unit
    const ScoreSmem lay = score_smem(D, G, B);
    int *nb = reinterpret_cast<int *>(smem + lay.nb);
    int *prefix = reinterpret_cast<int *>(smem + lay.prefix);
    int *misc = reinterpret_cast<int *>(smem + lay.misc);
    uint8_t *wb = smem + lay.warp0 + warp * lay.warp_bytes;
    uint8_t *ring = wb + lay.ring;
    uint8_t *qbuf = wb + lay.qbuf;
    uint64_t *bars = reinterpret_cast<uint64_t *>(wb + lay.bar);
    int4 *desc = reinterpret_cast<int4 *>(wb + lay.desc);
    const float NEG_INF = __int_as_float(0xff800000);

    build_item_space(p, nb, prefix, misc);
    if (lane == 0) {
        for (int s = 0; s < NSTAGE; ++s) mbar_init(&bars[s], 1);
        mbar_fence_init();
    }
    __syncthreads();  // the only CTA-wide barrier of the main path
    const int total_items = prefix[B];
    // Work schedule: about 80% of the units as one contiguous static block per warp (no
    // atomics, long sequential streams); the rest handed out from a global counter in
    // grabs that shrink from four units to one as the work runs out, so that the warps
    // finish together.  Each grab is requested one grab ahead, so its atomic never
    // stalls the warp.
    const int W = (int)gridDim.x * NWARP;
    const int gw = (int)blockIdx.x * NWARP + warp;
    const int Ks = (int)((long long)total_items * 4 / 5 / W);  // static units per warp
    const int dyn0 = Ks * W;                                    // the first dynamic unit

    // ---- producer state (warp-uniform; lane 0 issues the copies and the atomics)
    uint64_t policy = 0;
    const uint64_t keep = l2_policy_evict_last();  // the value stage reads these back
    int pend = 0;  // lane 0: the outstanding grab, first unit * 8 + size
    auto request = [&](int last) {
        if (lane == 0) {
            const int k = max(1, min(4, (total_items - last) / (2 * W)));
            pend = (dyn0 + atomicAdd(p.ctrl + CTRL_WORK, k)) * 8 + k;
        }
    };
    if (lane == 0) policy = l2_policy_evict_first();
    request(dyn0);
    int g_next = gw * Ks, g_end = g_next + Ks;  // the current grab: the static block first
    int pr_r = 0, pr_tile = 0, pr_ntiles = 0, pr_valid = 0, pr_grp = 0;
    long long pr_row0 = 0;
    bool pr_end = false;
    int pr_group = -1;          // (b * H_kv + g) of the last unit issued
    int q_issue0 = -1, q_issue1 = -1;  // sequence number of the tile carrying each q buffer
    int q_next = 0;             // the q buffer to use next
    int pr_seq = 0;             // sequence number of the next tile issued
    // position (b, g, r) of unit g_next, found by one search per grab and then stepped
    int ub = 0, ug = 0, ur = 0, uns = 1;
    auto seek = [&](int itm) {
        const Item x = decode_item(itm, prefix, nb, B, H_kv, L);
        ub = x.b;
        ug = x.g;
        ur = x.r;
        uns = x.ns;
    };
    auto step = [&]() {
        if (++ur == uns) {
            ur = 0;
            if (++ug == H_kv) {
                ug = 0;
                if (++ub < B) uns = nb[ub] > 0 ? (nb[ub] + L - 1) / L : 1;
            }
        }
    };
    if (g_next < g_end) seek(g_next);
    auto produce = [&](int slot, int cons_seq) {
        while (!pr_end && pr_tile == pr_ntiles) {
            if (g_next == g_end) {
                const int got = __shfl_sync(FULL, pend, 0);
                g_next = got >> 3;
                g_end = min(g_next + (got & 7), total_items);
                if (g_next >= total_items) {
                    pr_end = true;
                    break;
                }
                request(g_end);
                seek(g_next);
            }
            const int n = nb[ub];
            const int b = ub, g = ug, r = ur;
            ++g_next;
            step();
            if (n == 0) continue;  // empty rows are written by the value stage
            pr_r = r;
            pr_tile = 0;
            pr_valid = min(L, n - r * L);
            pr_ntiles = (pr_valid + T::KEYS - 1) / T::KEYS;
            pr_grp = b * H_kv + g;
            pr_row0 = (long long)pr_grp * p.n_max + (long long)r * L;
        }
        if (pr_end) {
            if (lane == 0) desc[slot] = make_int4(DESC_END, 0, 0, 0);
            return;
        }
        const int rows = min(T::KEYS, pr_valid - pr_tile * T::KEYS);
        int flags = 0;
        uint32_t qbytes = 0;
        int qb = 0;
        if (pr_tile == 0) {
            if (pr_grp != pr_group) {
                pr_group = pr_grp;
                flags |= TF_NEWQ;
                qb = (T::QBUF == 2) ? q_next : 0;
                const int busy = qb ? q_issue1 : q_issue0;
                // a staging buffer is free once the consumer has started the tile that carried it
                if (busy <= cons_seq) {
                    if (qb) q_issue1 = pr_seq; else q_issue0 = pr_seq;
                    if (T::QBUF == 2) q_next ^= 1;
                    flags |= qb << TF_QB_SHIFT;
                    qbytes = T::QBYTES;
                } else {
                    flags |= TF_QGLOBAL;
                }
            }
        }
        if (lane == 0) {
            desc[slot] = make_int4(pr_grp, (pr_r << 8) | pr_tile, rows, flags);
            const uint32_t bytes = (uint32_t)rows * C::ROWB;
            mbar_arrive_tx(&bars[slot], bytes + qbytes);
            bulk_g2s(ring + slot * T::BYTES, p.k + (pr_row0 + (long long)pr_tile * T::KEYS) * D, bytes,
                     &bars[slot], policy);
            // q[b][g*G .. g*G+G-1][:] is contiguous: the group's heads in one copy
            if (qbytes) bulk_g2s_plain(qbuf + qb * T::QBYTES, p.q + (size_t)pr_grp * G * D, qbytes, &bars[slot]);
        }
        ++pr_tile;
        ++pr_seq;
    };
    for (int s = 0; s < NSTAGE; ++s) produce(s, -1);

    // ---- consumer
    unsigned long long qp[G][8];
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
        // descriptor: group b*H_kv + g, (unit r << 8) | tile, rows, flags
        const int grpid = dsc.x, tile = dsc.y & 0xff, ur_c = dsc.y >> 8, rows = dsc.z, flags = dsc.w;
        if (flags & TF_NEWQ) {
            // the group's query heads: fp32 pairs of the lane's two 16-byte chunks per head
            const uint16_t *qg = (flags & TF_QGLOBAL)
                                     ? p.q + (size_t)grpid * G * D
                                     : reinterpret_cast<const uint16_t *>(qbuf + ((flags >> TF_QB_SHIFT) & 1) * T::QBYTES);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const uint4 a = *reinterpret_cast<const uint4 *>(qg + h * D + 8 * sub);
                const uint4 c = *reinterpret_cast<const uint4 *>(qg + h * D + 8 * (sub + C::P));
                const uint32_t wv[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) qp[h][i] = bf16x2_to_f32x2(wv[i]);
            }
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
        produce(slot, it);  // the tile and the query heads are in registers: refill the slot

        // ---- the chunk's maximum (log2 units) and its scale c_t
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
            ct[i] = ceilf(fminf(fmaxf(m, -16777216.f), 16777216.f));
        }

        // ---- weights (stored) and the chunk totals
        const size_t bh0 = (size_t)grpid * G;  // first query head of the group: b*H_q + g*G
        const size_t chunk = (size_t)ur_c * (L / CHUNK) + (size_t)tile;  // chunk index in the sequence
        float tot[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int h = C::head_of(lane, i);
            float *wrow = p.w + (bh0 + h) * p.n_pad + chunk * CHUNK;
            float acc = 0.f;
#pragma unroll
            for (int c = 0; c < NCALL; ++c) {
                const int key = c * C::KW + 2 * grp + C::key2_of(lane, i);
                if (key < rows) {
                    const float e = __fmaf_rn(sc[c][i], p.k2_lo, __fmaf_rn(sc[c][i], p.k2_hi, -ct[i]));
                    const float w = exp2f(e);
                    if (own) {
                        st_hint(wrow + key, w, keep);
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
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            if ((lane & C::SAME) == 0 && own) {
                const size_t ci = (bh0 + C::head_of(lane, i)) * p.nch + chunk;
                st_hint(p.ctot + ci, tot[i], keep);
                st_hint(p.cexp + ci, (int)ct[i], keep);
                st_hint(p.cmax + ci, tmx[i], keep);
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
