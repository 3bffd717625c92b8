// santa_dense.cuh -- dense split-K decode attention (the like-for-like baseline), sm_103a.
//
// Exact softmax attention o = sum_j p_j v_j, the value SANTA estimates ("Stochastic
// Sparse Attention for Memory-Bound Inference", abstract; the pages' baselines are
// split-K decode kernels).  The same persistent tile stream and score microkernel as the
// sampled kernel, but each stage carries the K and the V tile of 64 keys; every warp
// keeps an online softmax (running max, sum, and G x d partial outputs) over its keys;
// a split ends with a merge of the 8 warps into one partial (m, l, o) per query head,
// and the CTA that completes a group merges the group's splits into `out`.
#pragma once

#include "santa_sample.cuh"

namespace santa {

struct DenseSmem {
    int stage, bar, desc, misc, nb, prefix, pbuf, merge, total;
};

__host__ __device__ inline DenseSmem dense_smem(int D, int G, int B, int nstage)
{
    DenseSmem s{};
    const int P = D / 16, KW = 64 / P;
    int off = 0;
    s.stage = off; off += nstage * 2 * TILE_BYTES;
    s.bar = off; off += nstage * 8;
    s.desc = off; off += nstage * 16;
    s.misc = off; off += 16 * 4;
    s.nb = off; off += (int)align_up((size_t)B * 4, 16);
    s.prefix = off; off += (int)align_up((size_t)(B + 1) * 4, 16);
    s.pbuf = off; off += NWARP * KW * G * 8;
    off = (int)align_up((size_t)off, 16);
    s.merge = off; off += NWARP * G * D * 4 + NWARP * G * 2 * 4;
    s.total = off;
    return s;
}

template <int D, int G>
struct DenseCfg {
    using C = SampleCfg<D, G>;
    static constexpr int NSTAGE = 2;
    static constexpr int NPAIR = C::EPL / 2;   // output fp32 pairs per lane and head
    // a lane and slot that hold head h after the score reduction
    __host__ __device__ static constexpr int rep_lane(int h)
    {
        for (int l = 0; l < 32; ++l)
            for (int i = 0; i < C::NV; ++i)
                if (C::head_of(l, i) == h) return l;
        return 0;
    }
    __host__ __device__ static constexpr int rep_slot(int h)
    {
        for (int l = 0; l < 32; ++l)
            for (int i = 0; i < C::NV; ++i)
                if (C::head_of(l, i) == h) return i;
        return 0;
    }
    // both packed per head (lane in bits 0-7, slot above), evaluated by the compiler
    __host__ __device__ static constexpr unsigned long long rep_table()
    {
        unsigned long long t = 0;
        for (int h = 0; h < G; ++h)
            t |= (unsigned long long)(rep_lane(h) | (rep_slot(h) << 5)) << (8 * h);
        return t;
    }
    static constexpr unsigned long long REP = rep_table();
    __host__ __device__ static constexpr int lane_of(int h) { return (int)((REP >> (8 * h)) & 31); }
    __host__ __device__ static constexpr int slot_of(int h) { return (int)((REP >> (8 * h + 5)) & 7); }
};

template <int D, int G>
__global__ void __launch_bounds__(NT, (G <= 4 ? 2 : 1)) santa_dense_kernel(const Params p)
{
    using C = SampleCfg<D, G>;
    using DC = DenseCfg<D, G>;
    constexpr int NSTAGE = DC::NSTAGE;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sub = lane % C::P, grp = lane / C::P;
    const int B = p.B, H_kv = p.H_kv, H_q = p.H_q, L = p.L;
    const DenseSmem lay = dense_smem(D, G, B, NSTAGE);

    uint8_t *stage = smem + lay.stage;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + lay.bar);
    int4 *sdesc = reinterpret_cast<int4 *>(smem + lay.desc);
    int *misc = reinterpret_cast<int *>(smem + lay.misc);
    int *nb = reinterpret_cast<int *>(smem + lay.nb);
    int *prefix = reinterpret_cast<int *>(smem + lay.prefix);
    unsigned long long *pbuf = reinterpret_cast<unsigned long long *>(smem + lay.pbuf);
    float *mg_o = reinterpret_cast<float *>(smem + lay.merge);
    float *mg_ml = mg_o + NWARP * G * D;
    const float NEG_INF = __int_as_float(0xff800000);

    build_item_space(p, nb, prefix, misc);
    if (tid == 0) {
        for (int s = 0; s < NSTAGE; ++s) mbar_init(&bars[s], 1);
        mbar_fence_init();
    }
    __syncthreads();
    const int total_items = prefix[B];

    int pr_item = 0, pr_tile = 0, pr_ntiles = 0, pr_valid = 0, pr_next = 0;
    long long pr_row0 = 0;
    bool pr_end = false;
    uint64_t policy = 0;
    if (tid == 0) {
        policy = l2_policy_evict_first();
        pr_next = atomicAdd(p.ctrl + CTRL_WORK, 1);
    }
    auto produce = [&](int slot) {
        if (!pr_end && pr_tile == pr_ntiles) {
            const int it = pr_next;
            if (it < 0 || it >= total_items) {
                pr_end = true;
            } else {
                pr_next = atomicAdd(p.ctrl + CTRL_WORK, 1);
                const Item x = decode_item(it, prefix, nb, B, H_kv, L);
                pr_item = it;
                pr_tile = 0;
                if (x.n == 0) {
                    pr_ntiles = 0;
                    sdesc[slot] = make_int4(it, 0, 0, FLAG_ZERO);
                    mbar_arrive(&bars[slot]);
                    return;
                }
                pr_valid = min(L, x.n - x.r * L);
                pr_ntiles = (pr_valid + C::TK - 1) / C::TK;
                pr_row0 = ((long long)x.b * H_kv + x.g) * p.n_max + (long long)x.r * L;
            }
        }
        if (pr_end) {
            sdesc[slot] = make_int4(DESC_END, 0, 0, 0);
            mbar_arrive(&bars[slot]);
            return;
        }
        const int rows = min(C::TK, pr_valid - pr_tile * C::TK);
        const int flags = (pr_tile == pr_ntiles - 1) ? FLAG_LAST : 0;
        sdesc[slot] = make_int4(pr_item, pr_tile, rows, flags);
        const uint32_t bytes = (uint32_t)rows * C::ROWB;
        const long long row = pr_row0 + (long long)pr_tile * C::TK;
        mbar_arrive_tx(&bars[slot], 2 * bytes);
        bulk_g2s(stage + slot * 2 * TILE_BYTES, p.k + row * D, bytes, &bars[slot], policy);
        bulk_g2s(stage + slot * 2 * TILE_BYTES + TILE_BYTES, p.v + row * D, bytes, &bars[slot], policy);
        ++pr_tile;
    };
    if (tid == 0)
        for (int s = 0; s < NSTAGE; ++s) produce(s);

    unsigned long long qp[G][8];
    float m_w[G];                       // running maximum per head (log2 units), warp-uniform
    float l_l[C::NV];                   // this lane's share of the running sum, per score slot
    unsigned long long o2[G][DC::NPAIR];  // output partials: lane's EPL elements per head
    Item cur{0, 0, 0, 0, 1};
    bool aborted = false;
    int it = 0;

    for (;; ++it) {
        const int slot = it % NSTAGE;
        const uint32_t par = (uint32_t)(it / NSTAGE) & 1u;
        const bool ok = mbar_wait_bounded(&bars[slot], par, p.wait_ns);
        if (__syncthreads_or(!ok)) {
            aborted = true;
            break;
        }
        const int4 dsc = sdesc[slot];
        if (dsc.x == DESC_END) break;
        if (dsc.w & FLAG_ZERO) {
            const Item x = decode_item(dsc.x, prefix, nb, B, H_kv, L);
            for (int i = tid; i < G * D; i += NT) p.out[((size_t)x.b * H_q + x.g * G) * D + i] = 0.f;
            __syncthreads();
            if (tid == 0) produce(slot);
            continue;
        }
        const int tile = dsc.y, rows = dsc.z;
        if (tile == 0) {
            cur = decode_item(dsc.x, prefix, nb, B, H_kv, L);
            const uint16_t *qg = p.q + ((size_t)cur.b * H_q + (size_t)cur.g * G) * D;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const uint4 a = *reinterpret_cast<const uint4 *>(qg + h * D + 8 * sub);
                const uint4 c = *reinterpret_cast<const uint4 *>(qg + h * D + 8 * (sub + C::P));
                const uint32_t wv[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) qp[h][i] = bf16x2_to_f32x2(wv[i]);
                m_w[h] = NEG_INF;
#pragma unroll
                for (int j = 0; j < DC::NPAIR; ++j) o2[h][j] = 0ull;
            }
#pragma unroll
            for (int i = 0; i < C::NV; ++i) l_l[i] = 0.f;
        }
        const uint8_t *kt = stage + slot * 2 * TILE_BYTES;
        const uint8_t *vt = kt + TILE_BYTES;
        const int kwarp = warp * C::KW;
        const int kbase = kwarp + 2 * grp;
        float val[2 * G];
        tile_dots<D, G>(kt, kbase, sub, qp, val);
        float s2[C::NV];
#pragma unroll
        for (int i = 0; i < C::NV; ++i) {
            const int key = kbase + C::key2_of(lane, i);
            s2[i] = key < rows ? __fmul_rn(val[i], p.k2_hi) : NEG_INF;
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
        float m_new[G], alpha[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float mt = __shfl_sync(0xffffffffu, wm[DC::slot_of(h)], DC::lane_of(h));
            m_new[h] = fmaxf(m_w[h], mt);
            alpha[h] = (m_new[h] == NEG_INF) ? 1.f : exp2f(m_w[h] - m_new[h]);
            m_w[h] = m_new[h];
            const unsigned long long a2 = f32x2_pack(alpha[h], alpha[h]);
#pragma unroll
            for (int j = 0; j < DC::NPAIR; ++j) o2[h][j] = fmul2(o2[h][j], a2);
        }
        unsigned long long *pw = pbuf + warp * C::KW * G;
#pragma unroll
        for (int i = 0; i < C::NV; ++i) {
            const int h = C::head_of(lane, i);
            float mh = m_new[0], ah = alpha[0];
#pragma unroll
            for (int hh = 1; hh < G; ++hh) {
                mh = (h == hh) ? m_new[hh] : mh;
                ah = (h == hh) ? alpha[hh] : ah;
            }
            const float pr = (s2[i] == NEG_INF) ? 0.f : exp2f(s2[i] - mh);
            const bool own = (sub % C::REP) == 0;
            l_l[i] = __fmaf_rn(l_l[i], ah, own ? pr : 0.f);
            if (own) pw[(2 * grp + C::key2_of(lane, i)) * G + h] = f32x2_pack(pr, pr);
        }
        __syncwarp();
        const int nk = min(C::KW, rows - kwarp);
        for (int key = 0; key < nk; ++key) {
            const uint8_t *vrow = vt + (kwarp + key) * C::ROWB;
            unsigned long long vp[DC::NPAIR];
            if constexpr (C::EPL == 4) {
                const uint2 raw = *reinterpret_cast<const uint2 *>(vrow + 8 * lane);
                vp[0] = bf16x2_to_f32x2(raw.x);
                vp[1] = bf16x2_to_f32x2(raw.y);
            } else {
                const uint32_t raw = *reinterpret_cast<const uint32_t *>(vrow + 4 * lane);
                vp[0] = bf16x2_to_f32x2(raw);
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const unsigned long long pp = pw[key * G + h];
#pragma unroll
                for (int j = 0; j < DC::NPAIR; ++j) ffma2(o2[h][j], vp[j], pp);
            }
        }
        __syncthreads();
        if (tid == 0) produce(slot);

        if (!(dsc.w & FLAG_LAST)) continue;

        // ================= end of split: merge the warps into (m, l, o) per head
        const int b = cur.b, g = cur.g, r = cur.r;
        {
            float lsum[C::NV];
#pragma unroll
            for (int i = 0; i < C::NV; ++i) lsum[i] = l_l[i];
#pragma unroll
            for (int m = 1; m < 32; m <<= 1) {
                if (C::SAME & (unsigned)m) {
#pragma unroll
                    for (int i = 0; i < C::NV; ++i) lsum[i] = __fadd_rn(lsum[i], __shfl_xor_sync(0xffffffffu, lsum[i], m));
                }
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float lh = __shfl_sync(0xffffffffu, lsum[DC::slot_of(h)], DC::lane_of(h));
                if (lane == 0) {
                    mg_ml[(warp * G + h) * 2] = m_w[h];
                    mg_ml[(warp * G + h) * 2 + 1] = lh;
                }
#pragma unroll
                for (int j = 0; j < DC::NPAIR; ++j) {
                    const float2 f = f32x2_unpack(o2[h][j]);
                    mg_o[(warp * G + h) * D + C::EPL * lane + 2 * j] = f.x;
                    mg_o[(warp * G + h) * D + C::EPL * lane + 2 * j + 1] = f.y;
                }
            }
        }
        __syncthreads();
        for (int i = tid; i < G * D; i += NT) {
            const int h = i / D, dd = i % D;
            float M = NEG_INF;
#pragma unroll
            for (int w = 0; w < NWARP; ++w) M = fmaxf(M, mg_ml[(w * G + h) * 2]);
            float o = 0.f, l = 0.f;
#pragma unroll
            for (int w = 0; w < NWARP; ++w) {
                const float mw = mg_ml[(w * G + h) * 2];
                if (mw == NEG_INF) continue;
                const float f = exp2f(mw - M);
                o = __fmaf_rn(mg_o[(w * G + h) * D + dd], f, o);
                l = __fmaf_rn(mg_ml[(w * G + h) * 2 + 1], f, l);
            }
            const size_t bh = (size_t)b * H_q + g * G + h;
            p.dpart_o[(bh * p.ns_max + r) * D + dd] = o;
            if (dd == 0) {
                p.dpart_ml[(bh * p.ns_max + r) * 2] = M;
                p.dpart_ml[(bh * p.ns_max + r) * 2 + 1] = l;
            }
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            const int prev = atomicAdd(p.ctrl + CTRL_GROUPS + b * H_kv + g, 1);
            misc[MISC_LAST] = (prev == cur.ns - 1) ? 1 : 0;
        }
        __syncthreads();
        if (!misc[MISC_LAST]) continue;
        __threadfence();
        // ================= group epilogue: log-sum-exp merge of the splits
        const int ns = cur.ns;
        for (int i = tid; i < G * D; i += NT) {
            const int h = i / D, dd = i % D;
            const size_t bh = (size_t)b * H_q + g * G + h;
            float M = NEG_INF;
            for (int rr = 0; rr < ns; ++rr) M = fmaxf(M, __ldcg(p.dpart_ml + (bh * p.ns_max + rr) * 2));
            float o = 0.f, l = 0.f;
            for (int rr = 0; rr < ns; ++rr) {
                const float mr = __ldcg(p.dpart_ml + (bh * p.ns_max + rr) * 2);
                if (mr == NEG_INF) continue;
                const float f = exp2f(mr - M);
                o = __fmaf_rn(__ldcg(p.dpart_o + (bh * p.ns_max + rr) * D + dd), f, o);
                l = __fmaf_rn(__ldcg(p.dpart_ml + (bh * p.ns_max + rr) * 2 + 1), f, l);
            }
            p.out[bh * D + dd] = __fdiv_rn(o, l);
        }
        if (tid == 0) p.ctrl[CTRL_GROUPS + b * H_kv + g] = 0;
        __syncthreads();
    }

    if (aborted) {
        if (tid == 0) {
            set_dev_error(p.ctrl, DEV_TIMEOUT);
            for (int k = 0; k < NSTAGE; ++k) {
                const int j = it + k;
                mbar_wait_bounded(&bars[j % NSTAGE], (uint32_t)(j / NSTAGE) & 1u, p.wait_ns);
            }
        }
        __syncthreads();
    }
    if (tid == 0) {
        const int done = atomicAdd(p.ctrl + CTRL_EXIT, 1);
        if (done == (int)gridDim.x - 1) {
            p.ctrl[CTRL_WORK] = 0;
            p.ctrl[CTRL_EXIT] = 0;
        }
    }
}

}  // namespace santa
