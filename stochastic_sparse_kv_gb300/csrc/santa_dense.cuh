// santa_dense.cuh -- dense decode attention, the like-for-like baseline, sm_103a.
//
// Exact softmax attention o = sum_j p_j v_j: the quantity SANTA estimates ("Stochastic
// Sparse Attention for Memory-Bound Inference", abstract; the pages compare against
// split-K decode kernels).  Built like the score kernel of the sampled path, so that
// the comparison is like for like:
//
//  * persistent CTAs of 8 independent warps; a warp takes work units of UNIT keys of one
//    (b, g) -- a static contiguous block first, then shrinking grabs from a counter --
//    and streams K and V tiles of KEYS keys through its own ring of TMA bulk copies;
//  * per tile: the G query heads' scores (tile_dots), an online softmax per head (running
//    maximum m and sum l in log2 units, with rescaling when m grows), and p.V with the
//    tile's probabilities broadcast through shared memory; each lane owns D/32 output
//    dimensions of every head;
//  * at the end of a unit the warp writes its partial (m, l, o) per head; the warp that
//    completes the last unit of a group merges the group's partials into `out`.
#pragma once

#include "santa_sample.cuh"

namespace santa {

template <int D, int G>
struct DenseTile {
    static constexpr int KEYS = (D == 128) ? 16 : 32;  // keys per tile (a multiple of tile_dots' KW)
    static constexpr int KVB = KEYS * 2 * D;           // bytes of the tile's K (or V) part: 4 KB
    static constexpr int NSTAGE = 3;
    static constexpr int QBYTES = G * D * 2;
    static constexpr int UNIT = DENSE_UNIT;            // keys per work unit
    static constexpr int EPL = D / 32;                 // output dimensions per lane
};

struct DenseSmem {
    int nb, prefix, misc, warp0, warp_bytes, ring, qbuf, pbuf, bar, desc, total;
};

__host__ __device__ inline DenseSmem dense_smem(int D, int G, int B)
{
    const int keys = (D == 128) ? 16 : 32;
    const int kvb = keys * 2 * D;
    const int nstage = 3;
    DenseSmem s{};
    int off = 0;
    s.nb = off; off += (int)align_up((size_t)B * 4, 16);
    s.prefix = off; off += (int)align_up((size_t)(B + 1) * 4, 16);
    s.misc = off; off += 16 * 4;
    s.warp0 = (int)align_up((size_t)off, 128);
    int w = 0;
    s.ring = w; w += nstage * 2 * kvb;
    s.qbuf = w; w += G * D * 2;
    s.pbuf = w; w += keys * G * 4 + G * 4;  // the tile's p[key][head], then alpha[head]
    s.bar = w = (int)align_up((size_t)w, 8); w += nstage * 8;
    s.desc = w = (int)align_up((size_t)w, 16); w += nstage * 16;
    s.warp_bytes = (int)align_up((size_t)w, 128);
    s.total = s.warp0 + NWARP * s.warp_bytes;
    return s;
}

template <int D, int G>
__global__ void __launch_bounds__(NT, 1) santa_dense_kernel(const Params p)
{
    using C = SampleCfg<D, G>;
    using T = DenseTile<D, G>;
    constexpr int NSTAGE = T::NSTAGE;
    constexpr int NCALL = T::KEYS / C::KW;  // tile_dots calls per tile
    constexpr int NV = C::NV;
    constexpr int EPL = T::EPL;
    constexpr int L = T::UNIT;
    constexpr unsigned FULL = 0xffffffffu;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sub = lane % C::P, grp = lane / C::P;
    const int B = p.B, H_kv = p.H_kv, H_q = p.H_q;
    const DenseSmem lay = dense_smem(D, G, B);
    int *nb = reinterpret_cast<int *>(smem + lay.nb);
    int *prefix = reinterpret_cast<int *>(smem + lay.prefix);
    int *misc = reinterpret_cast<int *>(smem + lay.misc);
    uint8_t *wb = smem + lay.warp0 + warp * lay.warp_bytes;
    uint8_t *ring = wb + lay.ring;
    uint8_t *qbuf = wb + lay.qbuf;
    float *pk = reinterpret_cast<float *>(wb + lay.pbuf);  // [KEYS][G], then alpha[G]
    float *alpha_s = pk + T::KEYS * G;
    uint64_t *bars = reinterpret_cast<uint64_t *>(wb + lay.bar);
    int4 *desc = reinterpret_cast<int4 *>(wb + lay.desc);
    const float NEG_INF = __int_as_float(0xff800000);

    // the work units: UNIT keys per (b, g, r), counted per batch row like the score kernel's
    Params pu = p;
    pu.L = L;
    build_item_space(pu, nb, prefix, misc);
    if (lane == 0) {
        for (int s = 0; s < NSTAGE; ++s) mbar_init(&bars[s], 1);
        mbar_fence_init();
    }
    __syncthreads();  // the only CTA-wide barrier
    const int total_items = prefix[B];
    const int W = (int)gridDim.x * NWARP;
    const int gw = (int)blockIdx.x * NWARP + warp;
    const int Ks = (int)((long long)total_items * 4 / 5 / W);  // static units per warp
    const int dyn0 = Ks * W;

    // ---- producer (warp-uniform; lane 0 issues the copies and the atomics)
    uint64_t policy = 0;
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
    int pr_r = 0, pr_tile = 0, pr_ntiles = 0, pr_valid = 0, pr_grp = 0, pr_group = -1, pr_seq = 0;
    int q_issue = -1;  // sequence number of the tile that carried the staged query heads
    long long pr_row0 = 0;
    bool pr_end = false;
    int ub = 0, ug = 0, ur = 0, uns = 1;  // position of unit g_next
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
            if (n == 0) {  // an empty sequence: its group's outputs are zero
                float *o = p.out + ((size_t)b * H_q + (size_t)g * G) * D;
                for (int i = lane; i < G * D; i += 32) o[i] = 0.f;
                continue;
            }
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
        int flags = (pr_tile == pr_ntiles - 1) ? TF_LAST : 0;
        uint32_t qbytes = 0;
        if (pr_tile == 0 && pr_grp != pr_group) {
            pr_group = pr_grp;
            flags |= TF_NEWQ;
            // the staging buffer is free once the consumer has started the tile that carried it
            if (q_issue <= cons_seq) {
                q_issue = pr_seq;
                qbytes = T::QBYTES;
            } else {
                flags |= TF_QGLOBAL;
            }
        }
        if (lane == 0) {
            desc[slot] = make_int4(pr_grp, (pr_r << 8) | pr_tile, rows, flags);
            const uint32_t bytes = (uint32_t)rows * C::ROWB;
            const long long row = pr_row0 + (long long)pr_tile * T::KEYS;
            uint8_t *dst = ring + slot * 2 * T::KVB;
            mbar_arrive_tx(&bars[slot], 2 * bytes + qbytes);
            bulk_g2s(dst, p.k + row * D, bytes, &bars[slot], policy);
            bulk_g2s(dst + T::KVB, p.v + row * D, bytes, &bars[slot], policy);
            if (qbytes) bulk_g2s_plain(qbuf, p.q + (size_t)pr_grp * G * D, qbytes, &bars[slot]);
        }
        ++pr_tile;
        ++pr_seq;
    };
    for (int s = 0; s < NSTAGE; ++s) produce(s, -1);

    // ---- consumer
    unsigned long long qp[G][8];
    float m[NV], l[NV];   // per score slot (head): running maximum (log2 units) and sum
    float acc[G][EPL];    // this lane's output dimensions of every head
    auto reset_unit = [&]() {
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            m[i] = NEG_INF;
            l[i] = 0.f;
        }
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[h][e] = 0.f;
    };
    reset_unit();
    const bool own = (sub % C::REP) == 0;
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
        const int grpid = dsc.x, ur_c = dsc.y >> 8, rows = dsc.z, flags = dsc.w;
        if (flags & TF_NEWQ) {
            const uint16_t *qg = (flags & TF_QGLOBAL) ? p.q + (size_t)grpid * G * D
                                                       : reinterpret_cast<const uint16_t *>(qbuf);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const uint4 a = *reinterpret_cast<const uint4 *>(qg + h * D + 8 * sub);
                const uint4 c = *reinterpret_cast<const uint4 *>(qg + h * D + 8 * (sub + C::P));
                const uint32_t wv[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) qp[h][i] = bf16x2_to_f32x2(wv[i]);
            }
        }
        const uint8_t *kt = ring + slot * 2 * T::KVB;
        const uint8_t *vt = kt + T::KVB;

        // ---- scores, then the online softmax step of every head
        float sc[NCALL][NV];
#pragma unroll
        for (int c = 0; c < NCALL; ++c) {
            float val[2 * G];
            tile_dots<D, G>(kt, c * C::KW + 2 * grp, sub, qp, val);
#pragma unroll
            for (int i = 0; i < NV; ++i) sc[c][i] = val[i];
        }
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            float tm = NEG_INF;
#pragma unroll
            for (int c = 0; c < NCALL; ++c) {
                const int key = c * C::KW + 2 * grp + C::key2_of(lane, i);
                if (key < rows) tm = fmaxf(tm, __fmul_rn(sc[c][i], p.k2_hi));
            }
#pragma unroll
            for (int msk = 1; msk < 32; msk <<= 1)
                if (C::SAME & (unsigned)msk) tm = fmaxf(tm, __shfl_xor_sync(FULL, tm, msk));
            const float mn = fmaxf(m[i], tm);
            const float al = exp2f(m[i] - mn);  // 0 on the unit's first tile
            const int h = C::head_of(lane, i);
            float ps = 0.f;
#pragma unroll
            for (int c = 0; c < NCALL; ++c) {
                const int key = c * C::KW + 2 * grp + C::key2_of(lane, i);
                if (key < rows && own) {
                    const float pv = exp2f(__fmaf_rn(sc[c][i], p.k2_lo, __fmaf_rn(sc[c][i], p.k2_hi, -mn)));
                    pk[key * G + h] = pv;
                    ps = __fadd_rn(ps, pv);
                }
            }
#pragma unroll
            for (int msk = 1; msk < 32; msk <<= 1)
                if (C::SAME & (unsigned)msk) ps = __fadd_rn(ps, __shfl_xor_sync(FULL, ps, msk));
            l[i] = __fmaf_rn(l[i], al, ps);
            m[i] = mn;
            if ((lane & C::SAME) == 0 && own) alpha_s[h] = al;
        }
        __syncwarp();

        // ---- p.V: rescale, then add the tile's rows (this lane's EPL dimensions)
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float a = alpha_s[h];
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[h][e] = __fmul_rn(acc[h][e], a);
        }
        auto add_row = [&](int k) {
            float pv[G];
            if constexpr (G % 4 == 0) {
#pragma unroll
                for (int h4 = 0; h4 < G; h4 += 4) {
                    const float4 x = *reinterpret_cast<const float4 *>(pk + k * G + h4);
                    pv[h4] = x.x;
                    pv[h4 + 1] = x.y;
                    pv[h4 + 2] = x.z;
                    pv[h4 + 3] = x.w;
                }
            } else {
#pragma unroll
                for (int h = 0; h < G; ++h) pv[h] = pk[k * G + h];
            }
            float vv[EPL];
            if constexpr (EPL == 4) {
                const uint2 raw = *reinterpret_cast<const uint2 *>(vt + k * C::ROWB + 8 * lane);
                vv[0] = bf16lo_to_f32(raw.x);
                vv[1] = bf16hi_to_f32(raw.x);
                vv[2] = bf16lo_to_f32(raw.y);
                vv[3] = bf16hi_to_f32(raw.y);
            } else {
                const uint32_t raw = *reinterpret_cast<const uint32_t *>(vt + k * C::ROWB + 4 * lane);
                vv[0] = bf16lo_to_f32(raw);
                vv[1] = bf16hi_to_f32(raw);
            }
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < EPL; ++e) acc[h][e] = __fmaf_rn(pv[h], vv[e], acc[h][e]);
        };
        if (rows == T::KEYS) {  // full tiles: unrolled
#pragma unroll
            for (int k = 0; k < T::KEYS; ++k) add_row(k);
        } else {
            for (int k = 0; k < rows; ++k) add_row(k);
        }
        __syncwarp();
        produce(slot, it);  // K, V and the query heads are consumed: refill the slot

        // ---- end of a unit: its partial (m, l, o) per head; the last unit of a group merges
        if (flags & TF_LAST) {
            const size_t bh0 = (size_t)grpid * G;  // first query head of the group
#pragma unroll
            for (int i = 0; i < NV; ++i)
                if ((lane & C::SAME) == 0 && own) {
                    const size_t at = ((bh0 + C::head_of(lane, i)) * p.ns_max + ur_c) * 2;
                    p.dpart_ml[at] = m[i];
                    p.dpart_ml[at + 1] = l[i];
                }
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float *o = p.dpart_o + ((bh0 + h) * p.ns_max + ur_c) * D + EPL * lane;
#pragma unroll
                for (int e = 0; e < EPL; ++e) o[e] = acc[h][e];
            }
            reset_unit();
            __threadfence();
            __syncwarp();
            int done = 0;
            if (lane == 0) done = atomicAdd(p.ctrl + CTRL_GROUPS + grpid, 1) + 1;
            done = __shfl_sync(FULL, done, 0);
            const int nsg = (nb[grpid / H_kv] + L - 1) / L;
            if (done == nsg) {
                __threadfence();
                for (int h = 0; h < G; ++h) {
                    const size_t base = (bh0 + h) * p.ns_max;
                    float M = NEG_INF;
                    for (int u = lane; u < nsg; u += 32) M = fmaxf(M, __ldcg(p.dpart_ml + (base + u) * 2));
#pragma unroll
                    for (int msk = 16; msk >= 1; msk >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL, M, msk));
                    float o[EPL], lsum = 0.f;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) o[e] = 0.f;
#pragma unroll 4
                    for (int u = 0; u < nsg; ++u) {
                        const float f = exp2f(__ldcg(p.dpart_ml + (base + u) * 2) - M);
                        lsum = __fmaf_rn(f, __ldcg(p.dpart_ml + (base + u) * 2 + 1), lsum);
                        const float *ou = p.dpart_o + (base + u) * D + EPL * lane;
#pragma unroll
                        for (int e = 0; e < EPL; ++e) o[e] = __fmaf_rn(f, __ldcg(ou + e), o[e]);
                    }
                    float *dst = p.out + (bh0 + h) * D + EPL * lane;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) dst[e] = __fdiv_rn(o[e], lsum);
                }
                if (lane == 0) p.ctrl[CTRL_GROUPS + grpid] = 0;  // ready for the next call
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
    if (tid == 0) {
        const int done = atomicAdd(p.ctrl + CTRL_EXIT, 1);
        if (done == (int)gridDim.x - 1) {
            p.ctrl[CTRL_WORK] = 0;
            p.ctrl[CTRL_EXIT] = 0;
        }
    }
}

}  // namespace santa
