// santa_score.cuh -- SANTA score stage: scores, weights and per-chunk CDF pieces, sm_103a.
//
// "Stochastic Sparse Attention for Memory-Bound Inference" (abstract): the score stage
// reads all n_k cached keys and forms the post-softmax distribution from which the
// value stage samples.  This kernel streams the K cache (about 97% of the bytes of a
// sampled decode step) and is built so that nothing but that stream limits it:
//
//  * the contraction q . K^T runs on the tensor cores (tcgen05, bf16 inputs, fp32
//    accumulation in TMEM): a work unit is 128 consecutive keys of one KV head g of one
//    batch row b, and one unit is an M=128 x N=16 x K=d product whose N columns are the
//    group's G query heads (the rest padding).  The SIMT units keep only the softmax
//    epilogue (a handful of instructions per key instead of d*G/2 packed FMAs);
//  * persistent CTAs, one per SM, warp-specialised: one thread streams K tiles with
//    tiled TMA copies (128-byte swizzle, L2 evict-first) into a ring of stages, one
//    thread issues the MMAs, and two warpgroups of epilogue warps turn accumulators
//    into weights; mbarriers link the three (every wait bounded);
//  * a static contiguous block of units per CTA (about 60% of the work: 80% measured
//    1-2 us slower, 90% 10 us), then grabs from a global counter that shrink from four
//    units to one near the end, requested one grab ahead (grabs of one unit throughout
//    measured 30 us slower at B=16: runs of contiguous units matter);
//  * one epilogue warp handles one 32-key CDF chunk (its TMEM lane quarter), so chunks
//    are independent and need no state across units.
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
#include "santa_tcgen05.cuh"

namespace santa {

constexpr int SC_M = 128;              // keys per work unit = MMA rows
constexpr int SC_N = 16;               // MMA columns (query heads of the group, padded)
constexpr int SC_CHAIN = 1;            // K=16 MMA steps accumulated into one TMEM partial
constexpr int SC_TMEM_COLS = 512;      // all of TMEM: accumulators of every unit in flight
constexpr int SC_EPI_WARPS = 8;        // two warpgroups
constexpr int SC_WARP_PROD = 8;        // TMA producer
constexpr int SC_WARP_MMA = 9;         // MMA issuer, owner of the TMEM allocation
constexpr int SC_NT = 320;             // threads per CTA
constexpr int SC_BOX_ROWS = 32;        // rows per TMA box of a unit's tail (one CDF chunk)
constexpr int SC_RING_BYTES = 221184;  // stage ring (K + query tiles)

__host__ __device__ constexpr int score_halves(int D) { return D / 64; }  // 128-byte column blocks of a row
__host__ __device__ constexpr int score_kbytes(int D) { return score_halves(D) * SC_M * 128; }
__host__ __device__ constexpr int score_qbytes(int D) { return score_halves(D) * SC_N * 128; }
__host__ __device__ constexpr int score_stages(int D) { return SC_RING_BYTES / (score_kbytes(D) + score_qbytes(D)); }
// A unit's scores are the fp32 sum of D/(16*SC_CHAIN) partials, each SC_N TMEM columns;
// accumulators (units in flight between the MMA and the epilogue) fill the TMEM.
__host__ __device__ constexpr int score_chain(int D) { return SC_CHAIN < D / 16 ? SC_CHAIN : D / 16; }
__host__ __device__ constexpr int score_parts(int D) { return D / 16 / score_chain(D); }
__host__ __device__ constexpr int score_ucols(int D) { return score_parts(D) * SC_N; }
__host__ __device__ constexpr int score_nacc(int D)
{
    return SC_TMEM_COLS / score_ucols(D) < 32 ? SC_TMEM_COLS / score_ucols(D) : 32;
}

struct ScoreSmem {
    int kst, qst, bar, desc, adesc, tmem, nb, prefix, total;
};

// Byte offsets from the 1024-aligned base; `total` includes the alignment slack.
__host__ __device__ inline ScoreSmem score_smem(int D, int B)
{
    const int ns = score_stages(D), nacc = score_nacc(D);
    ScoreSmem s{};
    int off = 0;
    s.kst = off; off += ns * score_kbytes(D);
    s.qst = off; off += ns * score_qbytes(D);
    s.bar = off; off += (int)align_up((size_t)(2 * ns + 2 * nacc + 1) * 8, 16);
    s.desc = off; off += ns * 16;
    s.adesc = off; off += nacc * 16;
    s.tmem = off; off += 16;
    s.nb = off; off += (int)align_up((size_t)B * 4, 16);
    s.prefix = off; off += (int)align_up((size_t)(B + 1) * 4, 16);
    s.total = off + 1024;
    return s;
}

// A kernel's work-item space, built by one warp: nb[b] (checked lengths) and
// prefix[0..B] of the unit counts H_kv * ceil(n_b / L) (H_kv for n_b = 0).
__device__ __forceinline__ void warp_item_space(const Params &p, int L, int *nb, int *prefix)
{
    constexpr int PER = BMAX / 32;
    const int lane = threadIdx.x & 31;
    int sum = 0;
    bool bad = false;
#pragma unroll 8
    for (int i = 0; i < PER; ++i) {
        const int b = lane * PER + i;
        if (b < p.B) {
            int n = p.seq_lens[b];
            if (n < 0 || n > p.n_max) {
                bad = true;
                n = 0;
            }
            nb[b] = n;
            sum += p.H_kv * (n > 0 ? (n + L - 1) / L : 1);
        }
    }
    int x = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    int run = x - sum;
    for (int i = 0; i < PER; ++i) {
        const int b = lane * PER + i;
        if (b < p.B) {
            prefix[b] = run;
            run += p.H_kv * (nb[b] > 0 ? (nb[b] + L - 1) / L : 1);
        }
    }
    if (lane == 31) prefix[p.B] = x;
    if (bad && blockIdx.x == 0) set_dev_error(p.ctrl, DEV_BAD_SEQLEN);
    __syncwarp();
}

template <int D, int G>
__global__ void __launch_bounds__(SC_NT, 1)
    santa_score_kernel(const Params p, const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_kt,
                       const __grid_constant__ CUtensorMap tm_q)
{
    constexpr int NH = score_halves(D);
    constexpr int KB = SC_M * 128;   // one 128-byte column block of a K tile: 16 KB
    constexpr int QB = SC_N * 128;   // one column block of the query tile: 2 KB
    constexpr int NS = score_stages(D);
    constexpr int CH = score_chain(D);      // MMA steps per partial
    constexpr int NP = score_parts(D);      // partial sums per score
    constexpr int UCOLS = score_ucols(D);   // TMEM columns per unit
    constexpr int NACC = score_nacc(D);     // accumulators: unit j uses j % NACC
    static_assert(NACC >= 2 && NACC % 2 == 0 && NACC * UCOLS <= SC_TMEM_COLS, "TMEM accumulators");
    constexpr uint32_t IDESC = idesc_bf16_f32(SC_M, SC_N);
    constexpr unsigned FULL = 0xffffffffu;
    static_assert(G >= 1 && G <= 8 && SC_N >= G, "query heads per group");
    static_assert(NS >= 2, "stage ring");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const int B = p.B, H_kv = p.H_kv;
    const ScoreSmem lay = score_smem(D, B);
    uint8_t *kst = smem + lay.kst;
    uint8_t *qst = smem + lay.qst;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + lay.bar);
    uint64_t *empty = full + NS;
    uint64_t *tfull = empty + NS;
    uint64_t *tempty = tfull + NACC;
    uint64_t *drain = tempty + NACC;
    int4 *desc = reinterpret_cast<int4 *>(smem + lay.desc);
    int4 *adesc = reinterpret_cast<int4 *>(smem + lay.adesc);
    // [0] the TMEM address, [1] full phases the MMA thread consumed, [2] stages filled
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + lay.tmem);
    int *nb = reinterpret_cast<int *>(smem + lay.nb);
    int *prefix = reinterpret_cast<int *>(smem + lay.prefix);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float NEG_INF = __int_as_float(0xff800000);

    // ---- setup: TMEM, barriers, the work-item space, zero padding rows of the query tiles
    if (warp == SC_WARP_MMA) {
        tmem_alloc(tmem_slot, SC_TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == SC_WARP_PROD) {
        if (lane == 0) {
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
                mbar_init(&tfull[a], 2);      // the MMA commit and the issuing thread
                mbar_init(&tempty[a], 4);     // the four warps of the epilogue warpgroup
            }
            mbar_init(drain, 1);
            mbar_fence_init();
        }
        warp_item_space(p, SC_M, nb, prefix);
    }
    // rows G..SC_N-1 of every query tile: zero (the TMA copies fill rows 0..G-1)
    {
        constexpr int PIECES = (SC_N - G) * 8;  // 16-byte pieces per column block
        for (int i = tid; i < NS * NH * PIECES; i += SC_NT) {
            const int blk = i / PIECES, rem = i % PIECES;
            *reinterpret_cast<uint4 *>(qst + blk * QB + (G + rem / 8) * 128 + (rem % 8) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    if (tid == 0) SANTA_STAMP(blockIdx.x, 0);

    if (warp == SC_WARP_PROD) {
        // ================= producer: one thread streams K (and the group's queries)
        if (lane == 0) {
            const uint64_t policy = l2_policy_evict_first();
            const int total_items = prefix[B];
            const int W = (int)gridDim.x;
            const int Ks = (int)((long long)total_items * 3 / 5 / W);  // static units per CTA
            const int dyn0 = Ks * W;
            auto request = [&](int last) {
                const int k = max(1, min(4, (total_items - last) / (2 * W)));
                return (dyn0 + atomicAdd(p.ctrl + CTRL_WORK, k)) * 8 + k;
            };
            int pend = request(dyn0);
            int g_next = (int)blockIdx.x * Ks, g_end = g_next + Ks;
            int ub = 0, ug = 0, ur = 0, uns = 1;
            auto seek = [&](int itm) {
                const Item x = decode_item(itm, prefix, nb, B, H_kv, SC_M);
                ub = x.b;
                ug = x.g;
                ur = x.r;
                uns = x.ns;
            };
            if (g_next < g_end) seek(g_next);
            int i = 0;
            for (;; ++i) {
                // the next unit with keys, or the end of the work
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
                            if (++ub < B) uns = nb[ub] > 0 ? (nb[ub] + SC_M - 1) / SC_M : 1;
                        }
                    }
                    have = n > 0;  // empty rows are written by the value stage
                }
                const int s = i % NS;
                if (!mbar_wait_bounded(&empty[s], ((uint32_t)(i / NS) & 1u) ^ 1u, p.wait_ns)) {
                    set_dev_error(p.ctrl, DEV_TIMEOUT);
                    break;
                }
                if (!have) {
                    desc[s] = make_int4(DESC_END, 0, 0, 0);
                    mbar_arrive(&full[s]);
                    ++i;
                    break;
                }
                const int valid = min(SC_M, n - r * SC_M);
                const int grp = b * H_kv + g;
                desc[s] = make_int4(grp, r, valid, 0);
                const int row0 = grp * p.n_max + r * SC_M;
                uint8_t *kt = kst + s * NH * KB;
                if (valid == SC_M) {
                    // a full unit: one 128-row box per 128-byte column block
                    mbar_arrive_tx(&full[s], (uint32_t)(NH * KB + NH * G * 128));
#pragma unroll
                    for (int hf = 0; hf < NH; ++hf) tma_load_2d(kt + hf * KB, &tm_k, hf * 64, row0, &full[s], policy);
                } else {
                    // the sequence's last unit: 32-row boxes up to its last key
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
            SANTA_STAMP(blockIdx.x, 1);
        }
        __syncwarp();
    } else if (warp == SC_WARP_MMA) {
        // ================= MMA issuer: one thread; accumulator a = unit % NACC
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
                    // both epilogue warpgroups must see the end: units j and j + 1
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
                // step t = 4*hf + k covers d in [16t, 16t+16); partial t / CH takes CH steps
#pragma unroll
                for (int hf = 0; hf < NH; ++hf)
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int t = 4 * hf + k;
                        tc_mma_bf16(dt + (uint32_t)((t / CH) * SC_N), umma_desc_sw128(kaddr + hf * KB + k * 32),
                                    umma_desc_sw128(qaddr + hf * QB + k * 32), IDESC, (t % CH) != 0);
                    }
                tc_commit(&empty[s]);   // the stage may be refilled once these MMAs have read it
                tc_commit(&tfull[a]);   // the accumulator is ready
                mbar_arrive(&tfull[a]); // (releases adesc[a])
            }
            // every MMA complete before the allocation is released
            tc_commit(drain);
            mbar_wait_bounded(drain, 0u, DRAIN_NS);
        }
        __syncwarp();
    } else {
        // ================= epilogue: warp (e, w4) turns keys 32*w4.. of units e, e+2, ... into weights
        const int e = warp >> 2, w4 = warp & 3;
        const uint64_t keep = l2_policy_evict_last();  // the value stage reads these back
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
            const int grp = d.x, r = d.y, valid = d.z;
            const bool any = 32 * w4 < valid;  // warp-uniform
            // the NP partials of each head's score, summed in fp32 (round to nearest) as a tree
            float part[NP][G];
            if (any) {
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
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[a]);
            if (!any) continue;

            const int key = 32 * w4 + lane;   // key of the unit held by this lane
            const bool kv = key < valid;
            const size_t chunk = (size_t)r * (SC_M / CHUNK) + w4;
            const size_t bh0 = (size_t)grp * G;  // first query head of the group: b*H_q + g*G
            float sv[G], mx[G], ct[G], tot[G];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                sv[h] = part[0][h];
                mx[h] = kv ? __fmul_rn(sv[h], p.k2_hi) : NEG_INF;
            }
            // the chunk's maximum (log2 units) and its scale c_t
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
                for (int h = 0; h < G; ++h) mx[h] = fmaxf(mx[h], __shfl_xor_sync(FULL, mx[h], o));
            // weights (stored) and the chunk totals
#pragma unroll
            for (int h = 0; h < G; ++h) {
                ct[h] = ceilf(fminf(fmaxf(mx[h], -16777216.f), 16777216.f));
                float w = 0.f;
                if (kv) {
                    w = exp2f(__fmaf_rn(sv[h], p.k2_lo, __fmaf_rn(sv[h], p.k2_hi, -ct[h])));
                    st_hint(p.w + (bh0 + h) * p.n_pad + chunk * CHUNK + lane, w, keep);
                }
                tot[h] = w;
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
                for (int h = 0; h < G; ++h) tot[h] = __fadd_rn(tot[h], __shfl_xor_sync(FULL, tot[h], o));
            // lane h records head h's chunk
#pragma unroll
            for (int h = 0; h < G; ++h) {
                if (lane == h) {
                    const size_t ci = (bh0 + h) * p.nch + chunk;
                    st_hint(p.ctot + ci, tot[h], keep);
                    st_hint(p.cexp + ci, (int)ct[h], keep);
                    st_hint(p.cmax + ci, mx[h], keep);
                }
            }
        }
    }

    // ---- teardown: every MMA has completed (drained above); release TMEM.  After a
    // timeout, fills the MMA thread never consumed get a bounded wait to land first.
    tc_fence_before();
    __syncthreads();
    if (tid == 0) SANTA_STAMP(blockIdx.x, 2);
    if (warp == SC_WARP_PROD && lane == 0) {
        const int nfill = (int)tmem_slot[2];
        for (int f = (int)tmem_slot[1]; f < nfill; ++f)
            if (!mbar_wait_bounded(&full[f % NS], (uint32_t)(f / NS) & 1u, DRAIN_NS)) break;
    }
    if (warp == SC_WARP_MMA) {
        tc_fence_after();
        tmem_dealloc(tbase, SC_TMEM_COLS);
    }
    // The value stage is a programmatic dependent: let it launch only now (triggering at
    // the start measured ~9 us slower at B=16); it waits for the whole grid to complete.
    pdl_launch_dependents();
    if (tid == 0) SANTA_STAMP(blockIdx.x, 3);
    if (tid == 0) {
        const int done = atomicAdd(p.ctrl + CTRL_EXIT, 1);
        if (done == (int)gridDim.x - 1) {
            p.ctrl[CTRL_WORK] = 0;
            p.ctrl[CTRL_EXIT] = 0;
        }
    }
}

}  // namespace santa
