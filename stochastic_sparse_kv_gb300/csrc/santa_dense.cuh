// santa_dense.cuh -- dense decode attention, the like-for-like baseline, sm_103a.
//
// Exact softmax attention o = sum_j p_j v_j: the quantity SANTA estimates ("Stochastic
// Sparse Attention for Memory-Bound Inference", abstract; the pages compare against
// split-K decode kernels).  Built on the score kernel's machinery, so that the
// comparison is like for like:
//
//  * persistent CTAs, one per SM: one thread streams K, V and the group's query rows
//    with tiled TMA copies into a ring of stages (a stage = 128 keys of one (b, g)); one
//    thread issues q.K^T on the tensor cores (tcgen05, each K step into its own TMEM
//    partial); one warpgroup of four epilogue warps does the rest in fp32 on the CUDA
//    cores: the scores' online softmax per head, and p.V with V read from the stage
//    (each lane owns D/32 output dimensions of every head, p broadcast through shared
//    memory);
//  * the work items are splits of p.L keys (DENSE_UNIT, or 2 or 4 times that when the
//    problem has enough splits to keep every SM busy; a static contiguous block per CTA,
//    then shrinking grabs); the four warps combine their running (m, l, o) at the end of
//    a split and write one partial per (head, split);
//  * santa_dense_merge_kernel, a programmatic dependent launch, combines a head's
//    partials into `out` (the log-sum-exp merge of split-K decoding).
#pragma once

#include "santa_score.cuh"

namespace santa {

constexpr int DN_WARP_PROD = 4;        // TMA producer
constexpr int DN_WARP_MMA = 5;         // MMA issuer, owner of the TMEM allocation
constexpr int DN_NT = 192;             // threads per CTA: four epilogue warps, producer, MMA
constexpr int DN_RING_BYTES = 208896;  // K, V and query stages
constexpr int DN_HROUND = 4;           // heads combined per round at the end of a split
enum : int { DF_FIRST = 1, DF_LAST = 2 };  // descriptor flags: first / last subunit of a split

__host__ __device__ constexpr int dense_stages(int D)
{
    return DN_RING_BYTES / (2 * score_kbytes(D) + score_qbytes(D));
}

struct DenseSmem {
    int kst, vst, qst, bar, desc, adesc, tmem, pk, comb, nb, prefix, total;
};

// Byte offsets from the 1024-aligned base; `total` includes the alignment slack.
__host__ __device__ inline DenseSmem dense_smem(int D, int G, int B)
{
    const int ns = dense_stages(D), nacc = score_nacc(D);
    const int hr = G < DN_HROUND ? G : DN_HROUND;
    DenseSmem s{};
    int off = 0;
    s.kst = off; off += ns * score_kbytes(D);
    s.vst = off; off += ns * score_kbytes(D);
    s.qst = off; off += ns * score_qbytes(D);
    s.bar = off; off += (int)align_up((size_t)(2 * ns + 2 * nacc + 2) * 8, 16);
    s.desc = off; off += ns * 16;
    s.adesc = off; off += nacc * 16;
    s.tmem = off; off += 16;
    s.pk = off; off += 4 * 32 * G * 4;                                     // per warp: p[32 keys][G]
    s.comb = off; off += (int)align_up((size_t)4 * hr * (D + 2) * 4, 16);  // [warp][head][m, l, o[D]]
    s.nb = off; off += (int)align_up((size_t)B * 4, 16);
    s.prefix = off; off += (int)align_up((size_t)(B + 1) * 4, 16);
    s.total = off + 1024;
    return s;
}

template <int D, int G>
__global__ void __launch_bounds__(DN_NT, 1)
    santa_dense_kernel(const Params p, const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_kt,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_vt,
                       const __grid_constant__ CUtensorMap tm_q)
{
    constexpr int NH = score_halves(D);
    constexpr int KB = SC_M * 128;   // one 128-byte column block of a K or V tile: 16 KB
    constexpr int QB = SC_N * 128;   // one column block of the query tile: 2 KB
    constexpr int NS = dense_stages(D);
    constexpr int CH = score_chain(D);
    constexpr int NP = score_parts(D);
    constexpr int UCOLS = score_ucols(D);
    constexpr int NACC = score_nacc(D);
    constexpr int EPL = D / 32;              // output dimensions per lane
    const int L = p.L;                       // keys per split (one partial), a multiple of SC_M
    constexpr int HR = G < DN_HROUND ? G : DN_HROUND;
    constexpr uint32_t IDESC = idesc_bf16_f32(SC_M, SC_N);
    constexpr unsigned FULL = 0xffffffffu;
    static_assert(G >= 1 && G <= 8 && SC_N >= G, "query heads per group");
    static_assert(NS >= 2 && NACC >= 2, "stage ring and accumulators");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const int B = p.B, H_kv = p.H_kv;
    const DenseSmem lay = dense_smem(D, G, B);
    uint8_t *kst = smem + lay.kst;
    uint8_t *vst = smem + lay.vst;
    uint8_t *qst = smem + lay.qst;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + lay.bar);
    uint64_t *empty = full + NS;
    uint64_t *tfull = empty + NS;
    uint64_t *tempty = tfull + NACC;
    uint64_t *drain = tempty + NACC;
    uint64_t *wgbar = drain + 1;
    int4 *desc = reinterpret_cast<int4 *>(smem + lay.desc);
    int4 *adesc = reinterpret_cast<int4 *>(smem + lay.adesc);
    // [0] the TMEM address, [1] full phases the MMA thread consumed, [2] stages filled
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + lay.tmem);
    float *pk = reinterpret_cast<float *>(smem + lay.pk);
    float *comb = reinterpret_cast<float *>(smem + lay.comb);
    int *nb = reinterpret_cast<int *>(smem + lay.nb);
    int *prefix = reinterpret_cast<int *>(smem + lay.prefix);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float NEG_INF = __int_as_float(0xff800000);

    // ---- setup: TMEM, barriers, the work-item space, zero padding rows of the query tiles
    if (warp == DN_WARP_MMA) {
        tmem_alloc(tmem_slot, SC_TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == DN_WARP_PROD) {
        if (lane == 0) {
            tmem_slot[1] = 0;
            tmem_slot[2] = 0;
            tma_prefetch_map(&tm_k);
            tma_prefetch_map(&tm_kt);
            tma_prefetch_map(&tm_v);
            tma_prefetch_map(&tm_vt);
            tma_prefetch_map(&tm_q);
            for (int s = 0; s < NS; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], 4);  // the four epilogue warps, after their V reads
            }
            for (int a = 0; a < NACC; ++a) {
                mbar_init(&tfull[a], 2);   // the MMA commit and the issuing thread
                mbar_init(&tempty[a], 4);  // the four epilogue warps
            }
            mbar_init(drain, 1);
            mbar_init(wgbar, 4);           // the epilogue warps' own rendezvous
            mbar_fence_init();
        }
        warp_item_space(p, L, nb, prefix);
    }
    {
        constexpr int PIECES = (SC_N - G) * 8;  // 16-byte pieces per column block
        for (int i = tid; i < NS * NH * PIECES; i += DN_NT) {
            const int blk = i / PIECES, rem = i % PIECES;
            *reinterpret_cast<uint4 *>(qst + blk * QB + (G + rem / 8) * 128 + (rem % 8) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;

    if (warp == DN_WARP_PROD) {
        // ================= producer: one thread streams K, V and the group's queries
        if (lane == 0) {
            const uint64_t policy = l2_policy_evict_first();
            const int total_items = prefix[B];
            const int W = (int)gridDim.x;
            const int Ks = (int)((long long)total_items * 4 / 5 / W);  // static splits per CTA
            const int dyn0 = Ks * W;
            auto request = [&](int last) {
                const int k = max(1, min(4, (total_items - last) / (2 * W)));
                return (dyn0 + atomicAdd(p.ctrl + CTRL_WORK, k)) * 8 + k;
            };
            int pend = request(dyn0);
            int g_next = (int)blockIdx.x * Ks, g_end = g_next + Ks;
            int ub = 0, ug = 0, ur = 0, uns = 1;
            auto seek = [&](int itm) {
                const Item x = decode_item(itm, prefix, nb, B, H_kv, L);
                ub = x.b;
                ug = x.g;
                ur = x.r;
                uns = x.ns;
            };
            if (g_next < g_end) seek(g_next);
            int i = 0;  // stages filled
            bool stop = false;
            while (!stop) {
                // the next split with keys, or the end of the work
                int n = 0, b = 0, g = 0, r = 0;
                bool have = false;
                while (!have) {
                    if (g_next == g_end) {
                        g_next = pend >> 3;
                        g_end = min(g_next + (pend & 7), total_items);
                        if (g_next >= total_items) break;
                        pend = request(g_end);
                        seek(g_next);
                    }
                    n = nb[ub];
                    b = ub;
                    g = ug;
                    r = ur;
                    ++g_next;
                    if (++ur == uns) {
                        ur = 0;
                        if (++ug == H_kv) {
                            ug = 0;
                            if (++ub < B) uns = nb[ub] > 0 ? (nb[ub] + L - 1) / L : 1;
                        }
                    }
                    have = n > 0;  // empty rows: the merge kernel writes their zeros
                }
                const int vsplit = have ? min(L, n - r * L) : 0;
                const int nsub = have ? (vsplit + SC_M - 1) / SC_M : 1;
                for (int u = 0; u < nsub; ++u, ++i) {
                    const int s = i % NS;
                    if (!mbar_wait_bounded(&empty[s], ((uint32_t)(i / NS) & 1u) ^ 1u, p.wait_ns)) {
                        set_dev_error(p.ctrl, DEV_TIMEOUT);
                        stop = true;
                        break;
                    }
                    if (!have) {
                        desc[s] = make_int4(DESC_END, 0, 0, 0);
                        mbar_arrive(&full[s]);
                        ++i;
                        stop = true;
                        break;
                    }
                    const int valid = min(SC_M, vsplit - u * SC_M);
                    const int grp = b * H_kv + g;
                    desc[s] = make_int4(grp, r, valid, (u << 8) | (u == 0 ? DF_FIRST : 0) | (u == nsub - 1 ? DF_LAST : 0));
                    const int row0 = grp * p.n_max + r * L + u * SC_M;
                    uint8_t *kt = kst + s * NH * KB;
                    uint8_t *vt = vst + s * NH * KB;
                    if (valid == SC_M) {
                        mbar_arrive_tx(&full[s], (uint32_t)(2 * NH * KB + NH * G * 128));
#pragma unroll
                        for (int hf = 0; hf < NH; ++hf) {
                            tma_load_2d(kt + hf * KB, &tm_k, hf * 64, row0, &full[s], policy);
                            tma_load_2d(vt + hf * KB, &tm_v, hf * 64, row0, &full[s], policy);
                        }
                    } else {
                        const int nbox = (valid + SC_BOX_ROWS - 1) / SC_BOX_ROWS;
                        mbar_arrive_tx(&full[s], (uint32_t)(2 * nbox * NH * SC_BOX_ROWS * 128 + NH * G * 128));
                        for (int jb = 0; jb < nbox; ++jb)
#pragma unroll
                            for (int hf = 0; hf < NH; ++hf) {
                                const int off = hf * KB + jb * SC_BOX_ROWS * 128, y = row0 + jb * SC_BOX_ROWS;
                                tma_load_2d(kt + off, &tm_kt, hf * 64, y, &full[s], policy);
                                tma_load_2d(vt + off, &tm_vt, hf * 64, y, &full[s], policy);
                            }
                    }
#pragma unroll
                    for (int hf = 0; hf < NH; ++hf)
                        tma_load_2d_plain(qst + (s * NH + hf) * QB, &tm_q, hf * 64, grp * G, &full[s]);
                }
            }
            tmem_slot[2] = (uint32_t)i;
        }
        __syncwarp();
    } else if (warp == DN_WARP_MMA) {
        // ================= MMA issuer: one thread; accumulator a = stage fill % NACC
        if (lane == 0) {
            int j = 0;
            for (;; ++j) {
                const int s = j % NS, a = j % NACC;
                if (!mbar_wait_bounded(&full[s], (uint32_t)(j / NS) & 1u, p.wait_ns)) {
                    set_dev_error(p.ctrl, DEV_TIMEOUT);
                    break;
                }
                tmem_slot[1] = (uint32_t)(j + 1);
                const int4 d = desc[s];
                if (!mbar_wait_bounded(&tempty[a], ((uint32_t)(j / NACC) & 1u) ^ 1u, p.wait_ns)) {
                    set_dev_error(p.ctrl, DEV_TIMEOUT);
                    break;
                }
                tc_fence_after();
                adesc[a] = d;
                if (d.x == DESC_END) {
                    mbar_arrive(&tfull[a]);
                    mbar_arrive(&tfull[a]);
                    break;
                }
                const uint32_t kaddr = smem_u32(kst + s * NH * KB), qaddr = smem_u32(qst + s * NH * QB);
                const uint32_t dt = tbase + (uint32_t)(a * UCOLS);
#pragma unroll
                for (int hf = 0; hf < NH; ++hf)
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int t = 4 * hf + k;
                        tc_mma_bf16(dt + (uint32_t)((t / CH) * SC_N), umma_desc_sw128(kaddr + hf * KB + k * 32),
                                    umma_desc_sw128(qaddr + hf * QB + k * 32), IDESC, (t % CH) != 0);
                    }
                tc_commit(&tfull[a]);    // the scores are ready (the K tile has been read)
                mbar_arrive(&tfull[a]);  // (releases adesc[a])
            }
            tc_commit(drain);
            mbar_wait_bounded(drain, 0u, DRAIN_NS);
        }
        __syncwarp();
    } else {
        // ================= epilogue: warp w4 owns keys 32*w4.. of every subunit (its TMEM
        // lane quarter) and D/32 output dimensions of every head for those keys
        const int w4 = warp;
        float m[G], l[G], acc[G][EPL];   // running maximum (log2 units), this lane's sum, output
        auto reset = [&]() {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                m[h] = NEG_INF;
                l[h] = 0.f;
#pragma unroll
                for (int e = 0; e < EPL; ++e) acc[h][e] = 0.f;
            }
        };
        reset();
        uint32_t wg_phase = 0;
        // rendezvous of the four epilogue warps on an mbarrier (a bounded wait, unlike bar.sync)
        auto wg_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(wgbar);
            int ok = 1;
            if (lane == 0) ok = mbar_wait_bounded(wgbar, wg_phase, p.wait_ns) ? 1 : 0;
            __syncwarp();
            ok = __shfl_sync(FULL, ok, 0);
            wg_phase ^= 1u;
            return ok != 0;
        };
        // this lane's output dimensions d0 .. d0+EPL-1 inside a 128-byte swizzled V row
        const int d0 = EPL * lane;
        const int vhalf = d0 / 64, vpiece = (d0 % 64) / 8, vbyte = (d0 % 8) * 2;
        float *pkw = pk + w4 * 32 * G;
        for (int j = 0;; ++j) {
            const int a = j % NACC, s = j % NS;
            int ok = 1;
            if (lane == 0) ok = mbar_wait_bounded(&tfull[a], (uint32_t)(j / NACC) & 1u, p.wait_ns) ? 1 : 0;
            __syncwarp();
            ok = __shfl_sync(FULL, ok, 0);
            if (!ok) {
                if (lane == 0) set_dev_error(p.ctrl, DEV_TIMEOUT);
                break;
            }
            tc_fence_after();
            const int4 d = adesc[a];
            if (d.x == DESC_END) break;
            const int grp = d.x, r = d.y, valid = d.z, flags = d.w & 0xff;
            const bool any = 32 * w4 < valid;  // warp-uniform
            float sv[G];
            if (any) {
                float part[NP][G];
#pragma unroll
                for (int pp = 0; pp < NP; ++pp) {
                    uint32_t v[G];
                    tmem_ld32<G>(tbase + ((uint32_t)(32 * w4) << 16) + (uint32_t)(a * UCOLS + pp * SC_N), v);
#pragma unroll
                    for (int h = 0; h < G; ++h) part[pp][h] = __uint_as_float(v[h]);
                }
#pragma unroll
                for (int st = 1; st < NP; st <<= 1)
#pragma unroll
                    for (int pp = 0; pp + st < NP; pp += 2 * st)
#pragma unroll
                        for (int h = 0; h < G; ++h) part[pp][h] = __fadd_rn(part[pp][h], part[pp + st][h]);
#pragma unroll
                for (int h = 0; h < G; ++h) sv[h] = part[0][h];
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[a]);
            if (flags & DF_FIRST) reset();

            if (any) {
                const int key = 32 * w4 + lane;
                const bool kv = key < valid;
                // online softmax step per head (log2 units)
                float tm[G];
#pragma unroll
                for (int h = 0; h < G; ++h) tm[h] = kv ? __fmul_rn(sv[h], p.k2_hi) : NEG_INF;
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
                    for (int h = 0; h < G; ++h) tm[h] = fmaxf(tm[h], __shfl_xor_sync(FULL, tm[h], o));
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float mn = fmaxf(m[h], tm[h]);
                    const float al = exp2f(m[h] - mn);  // 0 on the split's first keys
                    const float pv = kv ? exp2f(__fmaf_rn(sv[h], p.k2_lo, __fmaf_rn(sv[h], p.k2_hi, -mn))) : 0.f;
                    l[h] = __fmaf_rn(l[h], al, pv);
#pragma unroll
                    for (int e = 0; e < EPL; ++e) acc[h][e] = __fmul_rn(acc[h][e], al);
                    m[h] = mn;
                    pkw[lane * G + h] = pv;
                }
                __syncwarp();
                // p.V over this warp's keys: each lane adds its EPL dimensions of every row
                const uint8_t *vt = vst + s * NH * KB + vhalf * KB;
                const int nk = min(32, valid - 32 * w4);
                auto add_row = [&](int k) {
                    const int row = 32 * w4 + k;
                    const uint8_t *src = vt + row * 128 + ((vpiece ^ (row & 7)) << 4) + vbyte;
                    float vv[EPL];
                    if constexpr (EPL == 4) {
                        const uint2 raw2 = *reinterpret_cast<const uint2 *>(src);
                        vv[0] = bf16lo_to_f32(raw2.x);
                        vv[1] = bf16hi_to_f32(raw2.x);
                        vv[2] = bf16lo_to_f32(raw2.y);
                        vv[3] = bf16hi_to_f32(raw2.y);
                    } else {
                        const uint32_t raw1 = *reinterpret_cast<const uint32_t *>(src);
                        vv[0] = bf16lo_to_f32(raw1);
                        vv[1] = bf16hi_to_f32(raw1);
                    }
                    float pv[G];
                    if constexpr (G % 4 == 0) {
#pragma unroll
                        for (int h4 = 0; h4 < G; h4 += 4) {
                            const float4 x = *reinterpret_cast<const float4 *>(pkw + k * G + h4);
                            pv[h4] = x.x;
                            pv[h4 + 1] = x.y;
                            pv[h4 + 2] = x.z;
                            pv[h4 + 3] = x.w;
                        }
                    } else {
#pragma unroll
                        for (int h = 0; h < G; ++h) pv[h] = pkw[k * G + h];
                    }
#pragma unroll
                    for (int h = 0; h < G; ++h)
#pragma unroll
                        for (int e = 0; e < EPL; ++e) acc[h][e] = __fmaf_rn(pv[h], vv[e], acc[h][e]);
                };
                if (nk == 32) {
#pragma unroll 8
                    for (int k = 0; k < 32; ++k) add_row(k);
                } else {
                    for (int k = 0; k < nk; ++k) add_row(k);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done with the stage's V

            if (flags & DF_LAST) {
                // the split's partial per head: the four warps' (m, l, o) combined in fp32
                const size_t bh0 = (size_t)grp * G;
                bool fine = true;
#pragma unroll
                for (int h0 = 0; h0 < G; h0 += HR) {
#pragma unroll
                    for (int hh = 0; hh < HR; ++hh) {
                        const int h = h0 + hh;
                        float lw = l[h];
#pragma unroll
                        for (int o = 16; o >= 1; o >>= 1) lw = __fadd_rn(lw, __shfl_xor_sync(FULL, lw, o));
                        float *cw = comb + (w4 * HR + hh) * (D + 2);
                        if (lane == 0) {
                            cw[0] = m[h];
                            cw[1] = lw;
                        }
#pragma unroll
                        for (int e = 0; e < EPL; ++e) cw[2 + d0 + e] = acc[h][e];
                    }
                    if (!(fine = wg_sync())) break;
                    const int t = 32 * w4 + lane;  // 0..127: one output dimension
#pragma unroll
                    for (int hh = 0; hh < HR; ++hh) {
                        const int h = h0 + hh;
                        float M = NEG_INF;
#pragma unroll
                        for (int w = 0; w < 4; ++w) M = fmaxf(M, comb[(w * HR + hh) * (D + 2)]);
                        float f[4];
#pragma unroll
                        for (int w = 0; w < 4; ++w) f[w] = exp2f(comb[(w * HR + hh) * (D + 2)] - M);
                        const size_t slot = (bh0 + h) * p.ns_max + r;
                        if (t < D) {
                            float o = 0.f;
#pragma unroll
                            for (int w = 0; w < 4; ++w) o = __fmaf_rn(f[w], comb[(w * HR + hh) * (D + 2) + 2 + t], o);
                            p.dpart_o[slot * D + t] = o;
                        }
                        if (t == 0) {
                            float ls = 0.f;
#pragma unroll
                            for (int w = 0; w < 4; ++w) ls = __fmaf_rn(f[w], comb[(w * HR + hh) * (D + 2) + 1], ls);
                            p.dpart_ml[slot * 2] = M;
                            p.dpart_ml[slot * 2 + 1] = ls;
                        }
                    }
                    if (!(fine = wg_sync())) break;  // the buffer is free again
                }
                if (!fine) {
                    if (lane == 0) set_dev_error(p.ctrl, DEV_TIMEOUT);
                    break;
                }
            }
        }
    }

    // ---- teardown: every MMA has completed (drained above); release TMEM.  After a
    // timeout, fills the MMA thread never consumed get a bounded wait to land first.
    tc_fence_before();
    __syncthreads();
    if (warp == DN_WARP_PROD && lane == 0) {
        const int nfill = (int)tmem_slot[2];
        for (int f = (int)tmem_slot[1]; f < nfill; ++f)
            if (!mbar_wait_bounded(&full[f % NS], (uint32_t)(f / NS) & 1u, DRAIN_NS)) break;
    }
    if (warp == DN_WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tbase, SC_TMEM_COLS);
    }
    // the merge kernel is a programmatic dependent; it waits for the whole grid
    pdl_launch_dependents();
    if (tid == 0) {
        const int done = atomicAdd(p.ctrl + CTRL_EXIT, 1);
        if (done == (int)gridDim.x - 1) {
            p.ctrl[CTRL_WORK] = 0;
            p.ctrl[CTRL_EXIT] = 0;
        }
    }
}

// The log-sum-exp merge of a head's split partials: o = sum_u 2^(m_u - M) o_u / sum_u
// 2^(m_u - M) l_u.  One CTA of MG_SLICES * D threads per (b, h_q): slice k adds the splits
// u = k mod MG_SLICES, and the slices' sums are added in slice order.  A head with no keys
// gets zeros.
constexpr int MG_SLICES = 4;

template <int D>
__global__ void __launch_bounds__(MG_SLICES * D) santa_dense_merge_kernel(const Params p)
{
    constexpr int NTM = MG_SLICES * D;
    __shared__ float f_s[NS_LIMIT];
    __shared__ float red[NTM / 32 + 1];
    __shared__ float part[MG_SLICES][D + 1];
    const int bh = blockIdx.x, b = bh / p.H_q, t = threadIdx.x;
    const int dim = t % D, slice = t / D;
    int n = p.seq_lens[b];
    if (n < 0 || n > p.n_max) n = 0;  // (flagged by the main kernel)
    const int nsg = (n + p.L - 1) / p.L;
    pdl_wait();  // the partials are complete and visible from here on
    if (nsg == 0) {
        if (t < D) store_out(p, (size_t)bh * D + t, 0.f);
        return;
    }
    const float *ml = p.dpart_ml + (size_t)bh * p.ns_max * 2;
    const float *po = p.dpart_o + (size_t)bh * p.ns_max * D;
    float M = __int_as_float(0xff800000);
    for (int u = t; u < nsg; u += NTM) {
        const float mu = __ldcg(ml + 2 * u);
        f_s[u] = mu;
        M = fmaxf(M, mu);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if ((t & 31) == 0) red[t >> 5] = M;
    __syncthreads();
    if (t == 0) {
        float x = red[0];
        for (int w = 1; w < NTM / 32; ++w) x = fmaxf(x, red[w]);
        red[NTM / 32] = x;
    }
    __syncthreads();
    M = red[NTM / 32];
    for (int u = t; u < nsg; u += NTM) f_s[u] = exp2f(f_s[u] - M);
    __syncthreads();
    float o = 0.f, ls = 0.f;
#pragma unroll 8
    for (int u = slice; u < nsg; u += MG_SLICES) {
        o = __fmaf_rn(f_s[u], __ldcg(po + (size_t)u * D + dim), o);
        ls = __fmaf_rn(f_s[u], __ldcg(ml + 2 * u + 1), ls);
    }
    part[slice][dim] = o;
    if (dim == 0) part[slice][D] = ls;
    __syncthreads();
    if (t < D) {
        float os = 0.f, lt = 0.f;
#pragma unroll
        for (int k = 0; k < MG_SLICES; ++k) {
            os = __fadd_rn(os, part[k][t]);
            lt = __fadd_rn(lt, part[k][D]);
        }
        store_out(p, (size_t)bh * D + t, __fdiv_rn(os, lt));
    }
}

}  // namespace santa
