// santa_cluster.cuh -- SANTA decode step in one pass for small batches, sm_103a.
//
// "Stochastic Sparse Attention for Memory-Bound Inference" (abstract): the score stage
// reads all n_k keys and forms the post-softmax distribution; the value stage samples
// S << n_k indices from it (stratified or systematic sampling) and gather-adds only those
// V rows, scaled by 1/S.  For a small batch the two-launch layout (santa_score.cuh, then
// santa_gather.cuh) is latency-bound: the whole value stage, a chain of round trips to
// memory per head, runs after the K stream, on data the score stage wrote to memory.
// This kernel does the whole step in one launch with the distribution kept on chip:
//
//  * one thread-block cluster of C CTAs per (batch row b, KV head g); CTA r streams a
//    contiguous run of 128-key units of that group with the score kernel's pipeline (TMA
//    into a ring of stages, tcgen05 q.K^T into TMEM, an epilogue that forms the fp32
//    weights and 32-key chunk data), and keeps the weights and chunk data of its keys in
//    shared memory instead of writing them out;
//  * then every CTA of the cluster takes part in the value stage of the group's G query
//    heads, exchanging only a few words per head over distributed shared memory:
//      1. per head, the CTA's largest chunk maximum and chunk scale go to every CTA;
//         after a cluster barrier each CTA knows the head's maximum M and scale 2^-C;
//      2. each CTA turns its chunk totals into 64-bit fixed point in the scale 2^-C and
//         re-scores, error-free, its keys within tau2 of M (their K rows are read again,
//         a few per CTA), patching weights and totals exactly as the two-launch path does;
//      3. each CTA's exclusive prefix over its chunks and its range total go to every CTA;
//         after a second barrier each CTA knows its offset in the head's CDF and Z;
//      4. each CTA draws all S points of each head, keeps the ones whose target t Z falls
//         in its own mass range, resolves them in shared memory (chunk, then key) and
//         writes their indices; the points of a key always land in one CTA;
//      5. each CTA gathers the distinct V rows of its points (one round trip) into
//         per-head partial sums, and the partial sums meet slice by slice: CTA k adds, in
//         rank order, its slice of ceil(D/C) dimensions of every CTA's partial sums after
//         a third barrier, and writes them to `out`.
//
// The score, weight, fixed-point and search arithmetic are those of the two-launch path,
// so the indices are the same (below the re-scoring caps); only the order of the fp32
// additions of the gather differs.  Every CTA reaches every cluster barrier: all other
// waits are bounded and no CTA leaves early.
#pragma once

#include <cooperative_groups.h>

#include "santa_score.cuh"

namespace santa {

constexpr int CL_NT = 384;    // 8 epilogue warps, the producer (8), the MMA issuer (9), two point warps
constexpr int CL_WARP_PTS = 10;  // first point warp: the points and the query heads, during the stream
constexpr int CL_PTS_BAR = 1;    // named barrier of the two point warps
constexpr int CL_HK = 128;    // heavy keys re-scored per head per CTA, at most
constexpr int CL_MAXC = 16;   // CTAs per cluster, at most
constexpr int CL_LWMAX = 4096;  // keys per CTA, at most (four 32-key chunks per lane in the prefix)
constexpr int CL_GTHREADS = 256;  // threads of the gather (warps 0-7)

// Stages of the ring: the most of these that fit beside the value stage's arrays.
__host__ __device__ constexpr int cluster_max_stages(int D) { return D == 128 ? 4 : 8; }
__host__ __device__ constexpr int cluster_min_stages(int D) { return D == 128 ? 3 : 6; }

struct ClusterSmem {
    int kst, qst, bar, desc, adesc, tmem, w, ctot, cmax, cexp, O, hot, hk, hkw, qf, tfx, sort, idx, lead, red, part,
        xmax, xcm, xtot, xpart, misc, total;
};

// Byte offsets from the 1024-aligned base; `total` includes the alignment slack.  LW: keys
// per CTA (a multiple of 128); C: CTAs per cluster; ns: stages of the ring.
__host__ __device__ inline ClusterSmem cluster_smem(int D, int G, int LW, int S, int mode, int C, int ns)
{
    const int nacc = score_nacc(D);
    const int DS = (D + C - 1) / C;  // output dimensions per CTA
    const int ncl = LW / CHUNK;  // chunks per CTA and head
    const int Sp = (mode == MODE_IID) ? next_pow2(S) : S;
    ClusterSmem s{};
    int off = 0;
    s.kst = off; off += ns * score_kbytes(D);
    s.qst = off; off += ns * score_qbytes(D);
    const int ring_end = off;
    // the value stage's scratch lives in the ring, which is free once the stream is over
    int v = 0;
    s.hot = v; v += G * ncl * 4;                                     // hot chunks per head
    s.hk = v; v += G * CL_HK * 4;                                    // heavy keys per head
    s.hkw = v; v += G * CL_HK * 4;                                   // their weights before re-scoring
    s.idx = v; v += (int)align_up((size_t)G * S * 4, 16);            // key per point (-1: another CTA's)
    s.lead = v; v += (int)align_up((size_t)(G * S + 2 * G) * 4, 16);  // distinct rows per head, counts
    s.red = v; v += CL_GTHREADS * 8 * 4;                             // gather partial sums [row group][head][D]
    s.part = v; v += G * D * 4;                                      // this CTA's partial sums [G][D]
    if (v > ring_end) off += v - ring_end;                           // (never, for the supported shapes)
    s.bar = off; off += (int)align_up((size_t)(2 * ns + 2 * nacc + 1) * 8, 16);
    s.desc = off; off += ns * 16;
    s.adesc = off; off += nacc * 16;
    s.tmem = off; off += 16;
    s.w = off; off += G * LW * 4;                        // [G][LW] weights
    s.ctot = off; off += G * ncl * 4;                    // [G][ncl] chunk totals
    s.cmax = off; off += G * ncl * 4;                    // chunk maxima (log2 units)
    s.cexp = off; off += G * ncl * 4;                    // chunk scales c_t
    s.O = (int)align_up((size_t)off, 16); off = s.O + G * ncl * 8;  // fixed-point totals, then prefix
    s.qf = off; off += G * D * 4;                        // the group's query heads in fp32
    s.tfx = (int)align_up((size_t)off, 16); off = s.tfx + G * S * 8;  // points as 64-bit fractions
    s.sort = off; off += (mode == MODE_IID) ? (int)align_up((size_t)G * Sp * 4, 16) : 0;  // iid: sort keys
    s.xmax = off; off += C * G * 4;                      // received: per CTA and head, max (key)
    s.xcm = off; off += C * G * 4;                       // ... and largest chunk scale
    s.xtot = (int)align_up((size_t)off, 8); off = s.xtot + C * G * 8;  // ... and range total
    s.xpart = (int)align_up((size_t)off, 16); off = s.xpart + C * G * DS * 4;  // ... partial sums of this CTA's slice [C][G][DS]
    s.misc = (int)align_up((size_t)off, 16); off = s.misc + 64 * 4;
    s.total = off + 1024;
    return s;
}

template <int D, int G>
__global__ void __launch_bounds__(CL_NT, 1)
    santa_cluster_kernel(const Params p, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_kt, const __grid_constant__ CUtensorMap tm_q)
{
    namespace cg = cooperative_groups;
    constexpr int NH = score_halves(D);
    constexpr int KB = SC_M * 128;
    constexpr int QB = SC_N * 128;
    const int NS = p.nstages;
    constexpr int CH = score_chain(D);
    constexpr int NP = score_parts(D);
    constexpr int UCOLS = score_ucols(D);
    constexpr int NACC = score_nacc(D);
    constexpr uint32_t IDESC = idesc_bf16_f32(SC_M, SC_N);
    constexpr unsigned FULL = 0xffffffffu;
    static_assert(G >= 1 && G <= 8, "query heads per group");
    static_assert(cluster_max_stages(D) * (score_kbytes(D) + score_qbytes(D)) <= SC_RING_BYTES, "stage ring");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    cg::cluster_group cl = cg::this_cluster();
    const int C = (int)cl.num_blocks();
    const int rk = (int)cl.block_rank();
    const int grp = (int)blockIdx.x / C;  // b * H_kv + g: clusters are runs of C consecutive CTAs
    const int b = grp / p.H_kv, g = grp % p.H_kv;
    const int LW = p.L;                   // keys per CTA (array stride)
    const int NCLM = LW / CHUNK;          // chunk-array stride
    const int S = p.S;
    const ClusterSmem lay = cluster_smem(D, G, LW, S, p.mode, C, NS);
    uint8_t *kst = smem + lay.kst;
    uint8_t *qst = smem + lay.qst;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + lay.bar);
    uint64_t *empty = full + NS;
    uint64_t *tfull = empty + NS;
    uint64_t *tempty = tfull + NACC;
    uint64_t *drain = tempty + NACC;
    int4 *desc = reinterpret_cast<int4 *>(smem + lay.desc);
    int4 *adesc = reinterpret_cast<int4 *>(smem + lay.adesc);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + lay.tmem);
    float *w_s = reinterpret_cast<float *>(smem + lay.w);
    float *ctot_s = reinterpret_cast<float *>(smem + lay.ctot);
    float *cmax_s = reinterpret_cast<float *>(smem + lay.cmax);
    int *cexp_s = reinterpret_cast<int *>(smem + lay.cexp);
    uint64_t *O_s = reinterpret_cast<uint64_t *>(smem + lay.O);
    int *hot = reinterpret_cast<int *>(smem + lay.hot);
    int *hk = reinterpret_cast<int *>(smem + lay.hk);
    float *hkw = reinterpret_cast<float *>(smem + lay.hkw);
    float *qf = reinterpret_cast<float *>(smem + lay.qf);
    uint64_t *tfx = reinterpret_cast<uint64_t *>(smem + lay.tfx);
    unsigned *sortk = reinterpret_cast<unsigned *>(smem + lay.sort);
    int *idx_s = reinterpret_cast<int *>(smem + lay.idx);
    int *lead = reinterpret_cast<int *>(smem + lay.lead);
    float *red = reinterpret_cast<float *>(smem + lay.red);
    float *part = reinterpret_cast<float *>(smem + lay.part);
    int *xmax = reinterpret_cast<int *>(smem + lay.xmax);
    int *xcm = reinterpret_cast<int *>(smem + lay.xcm);
    uint64_t *xtot = reinterpret_cast<uint64_t *>(smem + lay.xtot);
    float *xpart = reinterpret_cast<float *>(smem + lay.xpart);
    // misc: [0,8) max key per head, [8,16) scale per head, [16,24) hot chunks, [24,32)
    // heavy keys, [32,48) uint64 offset per head, [48,64) uint64 Z per head
    int *misc = reinterpret_cast<int *>(smem + lay.misc);
    uint64_t *offs = reinterpret_cast<uint64_t *>(misc + 32);
    uint64_t *zs = reinterpret_cast<uint64_t *>(misc + 48);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float NEG_INF = __int_as_float(0xff800000);
    if (tid == 0) SANTA_STAMP(blockIdx.x, 0);

    int n = p.seq_lens[b];
    if (n < 0 || n > p.n_max) {
        if (rk == 0 && g == 0 && tid == 0) set_dev_error(p.ctrl, DEV_BAD_SEQLEN);
        n = 0;
    }
    const int U = (n + SC_M - 1) / SC_M;   // units of the sequence
    const int Uc = (U + C - 1) / C;        // units per CTA (Uc * SC_M <= LW by the host's choice)
    const int u0 = min(rk * Uc, U), u1 = min(u0 + Uc, U);
    const int key0 = u0 * SC_M;            // first key of this CTA
    const int nkl = max(0, min(n, u1 * SC_M) - key0);  // keys of this CTA
    const int ncl = (nkl + CHUNK - 1) / CHUNK;         // chunks of this CTA

    // ---- setup: TMEM, barriers, zero padding rows of the query tiles, the query heads in fp32
    if (warp == SC_WARP_MMA) {
        tmem_alloc(tmem_slot, SC_TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == SC_WARP_PROD && lane == 0) {
        tmem_slot[1] = 0;
        tmem_slot[2] = 0;
        tma_prefetch_map(&tm_k);
        tma_prefetch_map(&tm_kt);
        tma_prefetch_map(&tm_q);
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < NACC; ++a) {
            mbar_init(&tfull[a], 2);
            mbar_init(&tempty[a], 4);
        }
        mbar_init(drain, 1);
        mbar_fence_init();
    }
    {
        constexpr int PIECES = (SC_N - G) * 8;
        for (int i = tid; i < NS * NH * PIECES; i += CL_NT) {
            const int blk = i / PIECES, rem = i % PIECES;
            *reinterpret_cast<uint4 *>(qst + blk * QB + (G + rem / 8) * 128 + (rem % 8) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    // first half of a cluster barrier: its wait, before the first store into another CTA's
    // shared memory, makes sure that every CTA of the cluster has started
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    if (tid == 0) SANTA_STAMP(blockIdx.x, 1);
    if (warp == SC_WARP_PROD) {
        // ================= producer: this CTA's units of the group, in order
        if (lane == 0) {
            const uint64_t policy = l2_policy_evict_first();
            int i = 0;
            for (int u = u0;; ++u, ++i) {
                const int s = i % NS;
                if (!mbar_wait_bounded(&empty[s], ((uint32_t)(i / NS) & 1u) ^ 1u, p.wait_ns)) {
                    set_dev_error(p.ctrl, DEV_TIMEOUT);
                    break;
                }
                if (u >= u1) {
                    desc[s] = make_int4(DESC_END, 0, 0, 0);
                    mbar_arrive(&full[s]);
                    ++i;
                    break;
                }
                const int valid = min(SC_M, n - u * SC_M);
                desc[s] = make_int4(grp, u - u0, valid, 0);
                const int row0 = grp * p.n_max + u * SC_M;
                uint8_t *kt = kst + s * NH * KB;
                if (valid == SC_M) {
                    mbar_arrive_tx(&full[s], (uint32_t)(NH * KB + NH * G * 128));
#pragma unroll
                    for (int hf = 0; hf < NH; ++hf) tma_load_2d(kt + hf * KB, &tm_k, hf * 64, row0, &full[s], policy);
                } else {
                    const int nbox = (valid + SC_BOX_ROWS - 1) / SC_BOX_ROWS;
                    mbar_arrive_tx(&full[s], (uint32_t)(nbox * NH * SC_BOX_ROWS * 128 + NH * G * 128));
                    for (int j = 0; j < nbox; ++j)
#pragma unroll
                        for (int hf = 0; hf < NH; ++hf)
                            tma_load_2d(kt + hf * KB + j * SC_BOX_ROWS * 128, &tm_kt, hf * 64, row0 + j * SC_BOX_ROWS,
                                        &full[s], policy);
                }
#pragma unroll
                for (int hf = 0; hf < NH; ++hf)
                    tma_load_2d_plain(qst + (s * NH + hf) * QB, &tm_q, hf * 64, grp * G, &full[s]);
            }
            tmem_slot[2] = (uint32_t)i;
            SANTA_STAMP(blockIdx.x, 2);
        }
        __syncwarp();
    } else if (warp == SC_WARP_MMA) {
        // ================= MMA issuer (as in the score kernel)
        if (lane == 0) {
            for (int j = 0;; ++j) {
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
                    const int a1 = (j + 1) % NACC;
                    if (mbar_wait_bounded(&tempty[a1], ((uint32_t)((j + 1) / NACC) & 1u) ^ 1u, p.wait_ns)) {
                        adesc[a1] = d;
                        mbar_arrive(&tfull[a1]);
                        mbar_arrive(&tfull[a1]);
                    } else {
                        set_dev_error(p.ctrl, DEV_TIMEOUT);
                    }
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
                tc_commit(&empty[s]);
                tc_commit(&tfull[a]);
                mbar_arrive(&tfull[a]);
            }
            tc_commit(drain);
            mbar_wait_bounded(drain, 0u, DRAIN_NS);
        }
        __syncwarp();
    } else if (warp < SC_EPI_WARPS) {
        // ================= epilogue (as in the score kernel), into shared memory
        const int e = warp >> 2, w4 = warp & 3;
        for (int u = 0;; ++u) {
            const int j = 2 * u + e, a = j % NACC;
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
            const int lu = d.y, valid = d.z;
            const bool any = 32 * w4 < valid;
            float part_[NP][G];
            if (any) {
#pragma unroll
                for (int pp = 0; pp < NP; ++pp) {
                    uint32_t v[G];
                    tmem_ld32<G>(tbase + ((uint32_t)(32 * w4) << 16) + (uint32_t)(a * UCOLS + pp * SC_N), v);
#pragma unroll
                    for (int h = 0; h < G; ++h) part_[pp][h] = __uint_as_float(v[h]);
                }
#pragma unroll
                for (int st = 1; st < NP; st <<= 1)
#pragma unroll
                    for (int pp = 0; pp + st < NP; pp += 2 * st)
#pragma unroll
                        for (int h = 0; h < G; ++h) part_[pp][h] = __fadd_rn(part_[pp][h], part_[pp + st][h]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[a]);
            if (!any) continue;
            const int key = 32 * w4 + lane;
            const bool kv = key < valid;
            const int lc = lu * (SC_M / CHUNK) + w4;  // local chunk
            float mx[G], ct[G], tot[G];
#pragma unroll
            for (int h = 0; h < G; ++h) mx[h] = kv ? __fmul_rn(part_[0][h], p.k2_hi) : NEG_INF;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
                for (int h = 0; h < G; ++h) mx[h] = fmaxf(mx[h], __shfl_xor_sync(FULL, mx[h], o));
#pragma unroll
            for (int h = 0; h < G; ++h) {
                ct[h] = ceilf(fminf(fmaxf(mx[h], -16777216.f), 16777216.f));
                float w = 0.f;
                if (kv) w = exp2f(__fmaf_rn(part_[0][h], p.k2_lo, __fmaf_rn(part_[0][h], p.k2_hi, -ct[h])));
                w_s[h * LW + lc * CHUNK + lane] = w;
                tot[h] = w;
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
                for (int h = 0; h < G; ++h) tot[h] = __fadd_rn(tot[h], __shfl_xor_sync(FULL, tot[h], o));
#pragma unroll
            for (int h = 0; h < G; ++h)
                if (lane == h) {
                    ctot_s[h * NCLM + lc] = tot[h];
                    cexp_s[h * NCLM + lc] = (int)ct[h];
                    cmax_s[h * NCLM + lc] = mx[h];
                }
        }
    }

    if (warp >= CL_WARP_PTS) {
        // ================= point warps, during the stream: the query heads in fp32 (for the
        // re-scoring) and the S points of each of the group's G heads (they do not depend
        // on the scores), as 64-bit fractions
        const int pt = tid - CL_WARP_PTS * 32;
        constexpr int NPT = CL_NT - CL_WARP_PTS * 32;
        for (int i = pt; i < G * D; i += NPT) qf[i] = __uint_as_float((uint32_t)p.q[((size_t)grp * G) * D + i] << 16);
        if (p.mode == MODE_IID) {
            const int Sp = next_pow2(S);
            for (int i = pt; i < G * Sp; i += NPT) {
                const int h = i / Sp, si = i % Sp;
                unsigned u = 0xffffffffu;
                if (si < S) {
                    uint64_t rnd[4];
                    philox_block(p.seed, (uint64_t)(si / 4), b, g * G + h, 3, rnd);
                    u = (unsigned)(rnd[si % 4] >> 32);
                }
                sortk[i] = u;
            }
            asm volatile("bar.sync %0, %1;" ::"n"(CL_PTS_BAR), "n"(NPT) : "memory");
            for (int kk = 2; kk <= Sp; kk <<= 1)
                for (int jj = kk >> 1; jj > 0; jj >>= 1) {
                    for (int i = pt; i < G * Sp; i += NPT) {
                        const int h = i / Sp, si = i % Sp, q2 = si ^ jj;
                        if (q2 > si) {
                            const bool asc = (si & kk) == 0;
                            const unsigned x = sortk[h * Sp + si], y = sortk[h * Sp + q2];
                            if ((x > y) == asc) {
                                sortk[h * Sp + si] = y;
                                sortk[h * Sp + q2] = x;
                            }
                        }
                    }
                    asm volatile("bar.sync %0, %1;" ::"n"(CL_PTS_BAR), "n"(NPT) : "memory");
                }
            for (int i = pt; i < G * S; i += NPT) tfx[i] = (uint64_t)sortk[(i / S) * Sp + i % S] << 32;
        } else {
            // each Philox block drawn once: one per head (systematic: the head's points share
            // its uniform) or one per four points (stratified); the raw words wait in the
            // point array until the points replace them (in integers, bit for bit the fp64
            // points of sample_point)
            const bool sys = p.mode == MODE_SYSTEMATIC;
            if (sys) {
                for (int h = pt; h < G; h += NPT) {
                    uint64_t rnd[4];
                    philox_block(p.seed, 0, b, g * G + h, 2, rnd);
                    tfx[h * S] = rnd[0];
                }
            } else {
                const int nb = (S + 3) / 4;
                for (int k = pt; k < G * nb; k += NPT) {
                    const int h = k / nb, jb = k % nb;
                    uint64_t rnd[4];
                    philox_block(p.seed, (uint64_t)jb, b, g * G + h, 1, rnd);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (4 * jb + e < S) tfx[h * S + 4 * jb + e] = rnd[e];
                }
            }
            asm volatile("bar.sync %0, %1;" ::"n"(CL_PTS_BAR), "n"(NPT) : "memory");
            uint64_t w0[G];
#pragma unroll
            for (int h = 0; h < G; ++h) w0[h] = sys ? tfx[h * S] : 0;
            asm volatile("bar.sync %0, %1;" ::"n"(CL_PTS_BAR), "n"(NPT) : "memory");
            const uint64_t rsb = (uint64_t)__double_as_longlong(p.rS);
            for (int i = pt; i < G * S; i += NPT) {
                const int h = i / S, si = i % S;
                uint64_t wh = 0;
#pragma unroll
                for (int k = 0; k < G; ++k)
                    if (k == h) wh = w0[k];
                tfx[i] = point_fraction(si, sys ? wh : tfx[i], rsb);
            }
        }
    }

    // ---- teardown of the score roles (as in the score kernel); the ring is then free for
    // the value stage's scratch, once the fills still in flight (after a timeout) have landed
    tc_fence_before();
    __syncthreads();
    if (tid == 0) SANTA_STAMP(blockIdx.x, 3);
    if (warp == SC_WARP_PROD && lane == 0) {
        const int nfill = (int)tmem_slot[2];
        for (int f = (int)tmem_slot[1]; f < nfill; ++f)
            if (!mbar_wait_bounded(&full[f % NS], (uint32_t)(f / NS) & 1u, DRAIN_NS)) break;
    }
    if (warp == SC_WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tbase, SC_TMEM_COLS);
    }
    __syncthreads();

    if (tid == 0) SANTA_STAMP(blockIdx.x, 4);
    // ================= value stage: every thread of the CTA
    if (tid < G) {
        misc[tid] = INT_MIN;      // below the key of every fp32 value
        misc[8 + tid] = INT_MIN;
        misc[16 + tid] = 0;
        misc[24 + tid] = 0;
    }
    __syncthreads();

    if (tid == 0) SANTA_STAMP(blockIdx.x, 5);
    // 1. this CTA's maximum and largest scale per head, to every CTA of the cluster
    for (int i = tid; i < G * ncl; i += CL_NT) {
        const int h = i / ncl, c = i % ncl;
        atomicMax(misc + h, fkey(cmax_s[h * NCLM + c]));
        atomicMax(misc + 8 + h, cexp_s[h * NCLM + c]);
    }
    __syncthreads();
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // (every CTA has started)
    for (int i = tid; i < C * G; i += CL_NT) {
        const int k = i / G, h = i % G;
        cl.map_shared_rank(xmax, k)[rk * G + h] = misc[h];
        cl.map_shared_rank(xcm, k)[rk * G + h] = misc[8 + h];
    }
    cl.sync();
    if (tid < G) {
        int mk = INT_MIN, cm = INT_MIN;
        for (int k = 0; k < C; ++k) {
            mk = max(mk, xmax[k * G + tid]);
            cm = max(cm, xcm[k * G + tid]);
        }
        misc[tid] = mk;
        misc[8 + tid] = cm;
    }
    __syncthreads();

    if (tid == 0) SANTA_STAMP(blockIdx.x, 6);
    // 2. fixed-point chunk totals in the head's scale 2^-C; hot chunks (maximum >= M - tau2)
    for (int i = tid; i < G * ncl; i += CL_NT) {
        const int h = i / ncl, c = i % ncl;
        const float thr = fkey_inv(misc[h]) - p.tau2;
        O_s[h * NCLM + c] = fixp(ctot_s[h * NCLM + c], FIX_F + cexp_s[h * NCLM + c] - misc[8 + h]);
        if (cmax_s[h * NCLM + c] >= thr) hot[h * NCLM + atomicAdd(misc + 16 + h, 1)] = c;
    }
    __syncthreads();
    //    heavy keys of the hot chunks (score >= M - tau2, read off their weights)
    for (int h = 0; h < G; ++h) {
        const int nh = misc[16 + h];
        const float thr = fkey_inv(misc[h]) - p.tau2;
        for (int q = tid; q < nh * CHUNK; q += CL_NT) {
            const int c = hot[h * NCLM + q / CHUNK], jl = c * CHUNK + q % CHUNK;
            if (jl < nkl) {
                const float wv = w_s[h * LW + jl];
                if (wv >= exp2f(thr - (float)cexp_s[h * NCLM + c])) {
                    const int pos = atomicAdd(misc + 24 + h, 1);
                    if (pos < CL_HK) {
                        hk[h * CL_HK + pos] = jl;
                        hkw[h * CL_HK + pos] = wv;
                    }
                }
            }
        }
    }
    __syncthreads();
    //    four lanes per heavy key re-score it error-free; weight rewritten, chunk total patched
    {
        int nk[G], tot = 0;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            nk[h] = min(misc[24 + h], CL_HK);
            tot += nk[h];
        }
        for (int t0 = 0; t0 < tot; t0 += CL_NT / 4) {  // (every lane runs every pass: they shuffle)
            const int t = t0 + tid / 4, part4 = tid & 3;
            const bool valid = t < tot;
            int h = 0, i = valid ? t : 0;
#pragma unroll
            for (int hh = 0; hh < G - 1; ++hh)
                if (h == hh && i >= nk[hh]) {
                    i -= nk[hh];
                    h = hh + 1;
                }
            const int jl = valid ? hk[h * CL_HK + i] : 0;
            const size_t row = (size_t)grp * p.n_max + (valid ? (size_t)(key0 + jl) : 0);
            float shi, slo;
            rescore_key_quad<D>(p.k + row * D, qf + h * D, part4, p.k2_hi, p.k2_lo, shi, slo);
            if (valid && part4 == 0) {
                const int c = jl / CHUNK;
                const int ctc = cexp_s[h * NCLM + c];
                const float wnew = exp2f(__fadd_rn(__fsub_rn(shi, (float)ctc), slo));
                w_s[h * LW + jl] = wnew;
                const int ee = FIX_F + ctc - misc[8 + h];
                const uint64_t dx = fixp(wnew, ee) - fixp(hkw[h * CL_HK + i], ee);
                if (dx) atomicAdd((unsigned long long *)(O_s + h * NCLM + c), (unsigned long long)dx);
            }
        }
    }
    __syncthreads();

    if (tid == 0) SANTA_STAMP(blockIdx.x, 7);
    // 3. exclusive prefix of this CTA's chunks per head (one warp per head, up to four
    //    consecutive chunks per lane); the range total to every CTA of the cluster
    if (warp < G) {
        const int h = warp;
        const int cpl = (ncl + 31) / 32;
        uint64_t v[4], sum = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int c = lane * cpl + e;
            v[e] = (e < cpl && c < ncl) ? O_s[h * NCLM + c] : 0ull;
            sum += v[e];
        }
        uint64_t x = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t y = __shfl_up_sync(FULL, x, o);
            if (lane >= o) x += y;
        }
        uint64_t ex = x - sum;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int c = lane * cpl + e;
            if (e < cpl && c < ncl) {
                O_s[h * NCLM + c] = ex;
                ex += v[e];
            }
        }
        const uint64_t total = __shfl_sync(FULL, x, 31);
        if (lane < C) cl.map_shared_rank(xtot, lane)[rk * G + h] = total;
    }
    cl.sync();
    if (tid < G) {
        uint64_t before = 0, z = 0;
        for (int k = 0; k < C; ++k) {
            const uint64_t t = xtot[k * G + tid];
            if (k < rk) before += t;
            z += t;
        }
        offs[tid] = before;
        zs[tid] = z;
    }
    __syncthreads();

    if (tid == 0) SANTA_STAMP(blockIdx.x, 8);
    // 4. the points of each head that fall in this CTA's mass range: T = t Z, then
    //    i = min{ j : W_j > T } by chunk (binary search on the prefix) and key (the chunk's
    //    weights), both in shared memory
    for (int i = tid; i < G * S; i += CL_NT) {
        const int h = i / S, s = i % S;
        const uint64_t Z = zs[h], base = offs[h];
        const uint64_t T = __umul64hi(tfx[i], Z);
        int j = -1;
        if (n > 0 && T >= base) {
            const uint64_t Tl = T - base;
            // (the range total is the prefix end: the last chunk's offset plus its total)
            int lo = 0, hi = ncl - 1;
            if (ncl > 0) {
                const uint64_t *Oh = O_s + h * NCLM;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (Oh[mid] <= Tl) lo = mid; else hi = mid - 1;
                }
            }
            if (ncl > 0 && Tl < xtot[rk * G + h]) {
                const int c = lo;
                const float rres = __fmul_rn(__ull2float_rn(Tl - O_s[h * NCLM + c]),
                                             exp2i(misc[8 + h] - cexp_s[h * NCLM + c] - FIX_F));
                const int j0 = c * CHUNK;
                const int jn = min(CHUNK, nkl - j0);
                const float4 *w4p = reinterpret_cast<const float4 *>(w_s + h * LW + j0);
                float wv[CHUNK];
#pragma unroll
                for (int k4 = 0; k4 < CHUNK / 4; ++k4) {
                    const float4 xv = w4p[k4];
                    wv[4 * k4] = xv.x;
                    wv[4 * k4 + 1] = xv.y;
                    wv[4 * k4 + 2] = xv.z;
                    wv[4 * k4 + 3] = xv.w;
                }
                const int pick = chunk_pick(wv, jn, rres);
                j = key0 + j0 + pick;
                if (p.idx_out) p.idx_out[((size_t)grp * G + h) * S + s] = j;
                const uint16_t *vrow = p.v + ((size_t)grp * p.n_max + j) * D;  // gathered below
                prefetch_l2(vrow);
                if (D * 2 > 128) prefetch_l2(vrow + 64);
            }
        }
        idx_s[h * S + s] = j;
        if (n == 0 && p.idx_out && (i % C) == rk) p.idx_out[((size_t)grp * G + h) * S + s] = -1;
    }
    __syncthreads();

    if (tid == 0) SANTA_STAMP(blockIdx.x, 9);
    // 5. the distinct V rows of this CTA's points (first occurrences, in point order; a key's
    //    points all land in this CTA, in one run), one warp per head: lead[h][k] = the k-th
    //    first occurrence, lead[G S + h] = their number, lead[G S + G + h] = 1 + the last point
    if (warp < G) {
        const int h = warp;
        int m = 0, last = -1;
        for (int s0 = 0; s0 < S; s0 += 32) {
            const int s = s0 + lane;
            const int j = s < S ? idx_s[h * S + s] : -1;
            const int jp = (s < S && s > 0) ? idx_s[h * S + s - 1] : -1;
            const bool first = j >= 0 && j != jp;
            const unsigned bl = __ballot_sync(FULL, first);
            if (first) lead[h * S + m + __popc(bl & ((1u << lane) - 1u))] = s;
            m += __popc(bl);
            const unsigned own = __ballot_sync(FULL, j >= 0);
            if (own) last = s0 + 31 - __clz(own);
        }
        if (lane == 0) {
            lead[G * S + h] = m;
            lead[G * S + G + h] = last + 1;
        }
    }
    __syncthreads();
    //    each distinct row loaded once and added times its count, by 16-byte pieces:
    //    thread = (row group, head, piece); the row groups' sums added in a fixed order
    {
        constexpr int NPC = D * 2 / 16;                 // 16-byte pieces per row
        constexpr int RG = CL_GTHREADS / (NPC * G);     // row groups per head
        const uint16_t *vg = p.v + (size_t)grp * p.n_max * D;
        if (tid < CL_GTHREADS) {
            const int piece = tid % NPC, h = (tid / NPC) % G, rg = tid / (NPC * G);
            const int nl = lead[G * S + h], send = lead[G * S + G + h];
            const int *lh = lead + h * S;
            float acc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = 0.f;
            for (int lb = rg; lb < nl; lb += 8 * RG) {
                uint4 rw[8];
                float cf[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int li = lb + u * RG;
                    cf[u] = 0.f;
                    rw[u] = make_uint4(0u, 0u, 0u, 0u);
                    if (li < nl) {
                        const int s = lh[li];
                        cf[u] = (float)((li + 1 < nl ? lh[li + 1] : send) - s);
                        rw[u] = *reinterpret_cast<const uint4 *>(vg + (size_t)idx_s[h * S + s] * D + 8 * piece);
                    }
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const uint32_t wv[4] = {rw[u].x, rw[u].y, rw[u].z, rw[u].w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        acc[2 * q] = __fmaf_rn(cf[u], bf16lo_to_f32(wv[q]), acc[2 * q]);
                        acc[2 * q + 1] = __fmaf_rn(cf[u], bf16hi_to_f32(wv[q]), acc[2 * q + 1]);
                    }
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) red[(rg * G + h) * D + 8 * piece + e] = acc[e];
        }
        __syncthreads();
        for (int i = tid; i < G * D; i += CL_NT) {
            const int h = i / D, dd = i % D;
            float sum = 0.f;
            for (int r = 0; r < RG; ++r) sum = __fadd_rn(sum, red[(r * G + h) * D + dd]);
            part[i] = sum;
        }
    }
    __syncthreads();
    if (tid == 0) SANTA_STAMP(blockIdx.x, 10);
    //    slice k (dimensions [k DS, (k+1) DS)) of every head's partial sums to CTA k
    const int DS = (D + C - 1) / C;
    if (DS % 4 == 0) {
        for (int i = tid; i < G * D / 4; i += CL_NT) {
            const int h = (4 * i) / D, dd = (4 * i) % D, k = dd / DS;
            *reinterpret_cast<float4 *>(cl.map_shared_rank(xpart, k) + (rk * G + h) * DS + dd % DS) =
                *reinterpret_cast<const float4 *>(part + 4 * i);
        }
    } else {
        for (int i = tid; i < G * D; i += CL_NT) {
            const int h = i / D, dd = i % D, k = dd / DS;
            cl.map_shared_rank(xpart, k)[(rk * G + h) * DS + dd % DS] = part[i];
        }
    }
    cl.sync();
    //    this CTA's slice of the outputs: the C partial sums in rank order, times 1/S
    for (int i = tid; i < G * DS; i += CL_NT) {
        const int h = i / DS, e = i % DS;
        if (rk * DS + e >= D) continue;
        float sum = 0.f;
        for (int k = 0; k < C; ++k) sum = __fadd_rn(sum, xpart[(k * G + h) * DS + e]);
        store_out(p, ((size_t)grp * G + h) * D + rk * DS + e, __fdiv_rn(sum, (float)S));
    }
    if (tid == 0) SANTA_STAMP(blockIdx.x, 11);
}

}  // namespace santa
