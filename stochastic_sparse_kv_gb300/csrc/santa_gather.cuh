// santa_gather.cuh -- SANTA value stage: sample points, CDF search, gather-add, sm_103a.
//
// "Stochastic Sparse Attention for Memory-Bound Inference" (abstract): sample S << n_k
// indices from the post-softmax distribution and aggregate only those value rows,
// scaled by 1/S.  One CTA per (batch row b, query head h), launched as a programmatic
// dependent of the score kernel: its CTAs start once every score CTA has finished (they
// cannot share an SM with one) and draw their points before the dependency wait.  The
// score kernel left, per 32-key
// chunk, the fp32 weights w_j in the chunk's scale 2^-c_t, the chunk total, c_t and the
// chunk's maximum score.  After the dependency wait the work is a few wide phases, each
// at most one round trip to memory, in integer or fp32 arithmetic only (written for a team
// of NTH threads synchronised by one barrier; the kernel's team is its whole CTA):
//   A. chunk data -> shared memory (left in global memory for very long sequences); the
//      maximum score M and the largest scale C over the sequence;
//   B. each chunk total as 64-bit fixed point in the global scale 2^-C,
//      G_c = round(tot_c 2^(FIX_F + c_t - C)); hot chunks: maximum >= M - tau2 (at most
//      HCAP: when more qualify, a histogram of the maxima keeps the hottest);
//   C. heavy keys: keys of hot chunks whose score is >= M - tau2 (read off their weights);
//   D. four lanes per heavy key re-score it error-free; its weight is rewritten and the
//      fixed-point change added to its chunk's G_c (integer atomics: exact, in any order).  The
//      heaviest keys' fp32 dot-product rounding would otherwise shift every later CDF
//      boundary;
//   E. the exact exclusive prefix O_c of the G_c (block scan), Z = the total;
//   F. one thread per point: T = t Z, i = min{ j : W_j > T } by chunk -> key, and (with
//      at most one point per thread) the selected V row prefetched into L2; then the
//      head's weights and chunk data, read for the last time, are discarded from L2
//      (never written back);
//   G. the distinct sampled rows (ordered compaction of the sorted list), each loaded
//      once -- 16-byte pieces spread over all threads, eight in flight per thread -- and
//      added times its count; out = sum / S (fp32, or rounded once to bf16).
#pragma once

#include <cooperative_groups.h>

#include "santa_sample.cuh"

namespace santa {

constexpr int NCH_SMEM = 4096;  // a head's chunk arrays stay in shared memory up to this many chunks
constexpr int NT_WIDE = 1024;   // the team of the wide variant (one CTA per SM: small batches)
constexpr int NCH_SMEM_WIDE = 10240;  // its chunk arrays stay in shared memory up to this many chunks
constexpr int NCH_WIDE_MIN = 2048;    // the wide variant for sequences of more chunks than this
__host__ __device__ constexpr int nch_smem_cap(int nth) { return nth > NT ? NCH_SMEM_WIDE : NCH_SMEM; }
constexpr int HCAP = 192;       // hot chunks re-scored per head, at most
constexpr int HBINS = 256;      // histogram bins that pick the hottest HCAP chunks
constexpr int XDEDUP_MAX = 8192;  // G * S up to which the group's heads share their V loads
// value-stage kernel variants (bits): group dedup, i.i.d. points, and the wide team of
// NT_WIDE threads for batches of at most one head per SM (not with group dedup)
enum : int { GATHER_XD = 1, GATHER_IID = 2, GATHER_WIDE = 4 };

// Whether the value stage can run as clusters of the group's G heads that load each
// distinct V row once for all of them (on request: SANTA_GROUP_DEDUP; the host then
// launches clusters of G and sets Params::xdedup).
__host__ __device__ inline bool gather_xdedup(int G, int S) { return G > 1 && G * S <= XDEDUP_MAX; }
constexpr int HKCAP = 512;      // heavy keys re-scored per head, at most

// misc words of the value stage (GM_SCAN: the block scan's NTH/32 + 1 64-bit words)
enum : int { GM_MAX = 0, GM_CMAX = 1, GM_NHOT = 2, GM_NHV = 3, GM_CNT = 4, GM_SCAN = 8 };

struct GatherSmem {
    int t, O, tot, ce, cm, hot, hv, hvw, hist, idx, lead, acc, qf, all, own, recv, misc, total;
};

// Shared memory of one team's value stage (nth threads; xd: the group-deduplicating
// gather of the two-pass kernel).
__host__ __device__ inline GatherSmem gather_smem(int D, int G, int S, int nch_used, int mode, bool xd, int nth = NT)
{
    GatherSmem s{};
    const int Sp = (mode == MODE_IID) ? next_pow2(S) : S;
    const int ncs = nch_used <= nch_smem_cap(nth) ? nch_used : 0;
    int off = 0;
    s.t = off; off += S * 8;
    s.O = off; off += ncs * 8;
    s.tot = off; off = (int)align_up((size_t)off + ncs * 4, 16);
    s.ce = off; off = (int)align_up((size_t)off + ncs * 4, 16);
    s.cm = off; off = (int)align_up((size_t)off + ncs * 4, 16);
    s.hot = off; off = (int)align_up((size_t)off + HCAP * 4, 16);
    s.hv = off; off = (int)align_up((size_t)off + HKCAP * 4, 16);
    s.hvw = off; off = (int)align_up((size_t)off + HKCAP * 4, 16);
    s.hist = off; off = (int)align_up((size_t)off + HBINS * 4, 16);
    s.idx = off; off = (int)align_up((size_t)off + Sp * 4, 16);
    // G's arrays overlay what F read for the last time, so that four CTAs fit on an SM up to
    // S = 2048: the distinct-row list over the points ((S + 1) * 4 <= S * 8 bytes), the
    // per-thread partial sums of the gather (8 dims each) over the chunk arrays, when these
    // are large enough
    s.lead = s.t;
    const int accb = nth * 8 * 4;
    if (s.hot - s.O >= accb) {
        s.acc = s.O;
    } else {
        s.acc = off;
        off += accb;
    }
    s.qf = off; off += D * 4;
    // group dedup: the group's G lists, then (after them) the partial sums of the NWARP warps,
    // over the points and chunk arrays when these are large enough (the lists are pushed
    // only once every CTA of the group is past F); the partial sums received, their own
    const int xall = xd ? max(G * S * 4, NWARP * G * D * 4) : 0;
    if (s.hot - s.t >= xall) {
        s.all = s.t;
    } else {
        s.all = off;
        off = (int)align_up((size_t)off + xall, 16);
    }
    s.own = s.all;
    s.recv = off; off = (int)align_up((size_t)off + (xd ? G * D * 4 : 0), 16);
    s.misc = off; off += (int)align_up((size_t)max(32, GM_SCAN + 2 * (nth / 32 + 1)) * 4, 16);
    s.total = (int)align_up((size_t)off, 128);
    return s;
}


// Barrier of a team of NTH threads: the whole CTA (BAR = 0) or named barrier BAR.
template <int BAR, int NTH>
__device__ __forceinline__ void team_sync()
{
    if constexpr (BAR == 0)
        __syncthreads();
    else
        asm volatile("bar.sync %0, %1;" ::"n"(BAR), "n"(NTH) : "memory");
}

// Exclusive scan of one int per team thread; the team total via *total.
template <int BAR, int NTH>
__device__ __forceinline__ int team_excl_scan(int v, int tid, int *scratch /*NTH/32+1 ints*/, int *total)
{
    constexpr int NW = NTH / 32;
    const int lane = tid & 31, warp = tid >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    team_sync<BAR, NTH>();
    if (tid == 0) {
        int acc = 0;
        for (int w = 0; w < NW; ++w) {
            const int t = scratch[w];
            scratch[w] = acc;
            acc += t;
        }
        scratch[NW] = acc;
    }
    team_sync<BAR, NTH>();
    const int res = scratch[warp] + x - v;
    *total = scratch[NW];
    team_sync<BAR, NTH>();
    return res;
}

// The checked length of batch row b (out-of-range values count as 0; the score stage
// flags them in the device error word).
__device__ __forceinline__ int value_len(const Params &p, int b)
{
    const int n = p.seq_lens[b];
    return (n < 0 || n > p.n_max) ? 0 : n;
}

// A head of an empty row: out = 0, indices -1.
template <int D, int NTH>
__device__ __forceinline__ void value_empty(const Params &p, int bh, int tid)
{
    for (int i = tid; i < D; i += NTH) store_out(p, (size_t)bh * D + i, 0.f);
    if (p.idx_out)
        for (int i = tid; i < p.S; i += NTH) p.idx_out[(size_t)bh * p.S + i] = -1;
}

// 0. The points (independent of the scores), the query head in fp32 and the team's
// counters.  Needs no score-stage result.
template <int D, int G, int NTH, int BAR, bool IID>
__device__ __forceinline__ void value_prologue(const Params &p, int bh, uint8_t *smem, const GatherSmem &lay, int tid)
{
    const int H_q = p.H_q, S = p.S;
    const int b = bh / H_q, h = bh % H_q;
    uint64_t *tfx = reinterpret_cast<uint64_t *>(smem + lay.t);  // points as 64-bit fractions
    int *idx = reinterpret_cast<int *>(smem + lay.idx);
    float *qf = reinterpret_cast<float *>(smem + lay.qf);
    int *misc = reinterpret_cast<int *>(smem + lay.misc);
    const int Sp = IID ? next_pow2(S) : S;
    if constexpr (IID) {
        unsigned *uk = reinterpret_cast<unsigned *>(idx);
        // one Philox block per four points, drawn once (thread j draws block j); the
        // padding up to a power of two sorts last
        for (int j = tid; 4 * j < Sp; j += NTH) {
            uint64_t rnd[4] = {0, 0, 0, 0};
            if (4 * j < S) philox_block(p.seed, (uint64_t)j, b, h, 3, rnd);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int s = 4 * j + e;
                if (s < Sp) uk[s] = s < S ? (unsigned)(rnd[e] >> 32) : 0xffffffffu;
            }
        }
        team_sync<BAR, NTH>();
        for (int kk = 2; kk <= Sp; kk <<= 1)
            for (int jj = kk >> 1; jj > 0; jj >>= 1) {
                for (int s = tid; s < Sp; s += NTH) {
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
                team_sync<BAR, NTH>();
            }
        for (int s = tid; s < S; s += NTH) tfx[s] = (uint64_t)uk[s] << 32;  // u = x 2^-32 exactly
    } else {
        // The Philox blocks, each drawn once: one per head (systematic: every point shares
        // its uniform), or one per four points (stratified: the raw words wait in the point
        // array until each thread replaces its own with its point).  Then each point as a
        // 64-bit fraction, bit for bit the fp64 point of sample_point, in integers.
        const bool sys = p.mode == MODE_SYSTEMATIC;
        uint64_t *w0 = reinterpret_cast<uint64_t *>(misc + GM_SCAN);
        if (sys) {
            if (tid == 0) {
                uint64_t rnd[4];
                philox_block(p.seed, 0, b, h, 2, rnd);
                *w0 = rnd[0];
            }
        } else {
            for (int j = tid; 4 * j < S; j += NTH) {
                uint64_t rnd[4];
                philox_block(p.seed, (uint64_t)j, b, h, 1, rnd);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (4 * j + e < S) tfx[4 * j + e] = rnd[e];
            }
        }
        team_sync<BAR, NTH>();
        const uint64_t rsb = (uint64_t)__double_as_longlong(p.rS);
        for (int s = tid; s < S; s += NTH) tfx[s] = point_fraction(s, sys ? *w0 : tfx[s], rsb);
    }
    for (int i = tid; i < D; i += NTH) qf[i] = __uint_as_float((uint32_t)p.q[(size_t)bh * D + i] << 16);
    if (tid == 0) {
        misc[GM_MAX] = INT_MIN;  // below the key of every fp32 value
        misc[GM_CMAX] = INT_MIN;
        misc[GM_NHOT] = 0;
        misc[GM_NHV] = 0;
        misc[GM_CNT] = 0;
    }
}

// Phases A-G of head bh (n >= 1 keys), after the team has synchronised past the wait
// for the score stage's results.  XD: the group-deduplicating gather (two-pass kernel
// launched as clusters of the group's G heads).
template <int D, int G, int NTH, int BAR, bool XD>
__device__ __forceinline__ void value_main(const Params &p, int bh, int n, uint8_t *smem, const GatherSmem &lay,
                                           int tid)
{
    constexpr int EPL = D / 32;  // V elements per lane
    constexpr int NW = NTH / 32;
    const int lane = tid & 31, warp = tid >> 5;
    const unsigned FULL = 0xffffffffu;
    const int H_q = p.H_q, S = p.S;
    const int b = bh / H_q, h = bh % H_q, g = h / G;
    (void)h;
    const int nchn = (n + CHUNK - 1) / CHUNK;  // chunks of this sequence
    const bool in_smem = p.nch <= nch_smem_cap(NTH);
    const size_t bhc = (size_t)bh * p.nch;
    uint64_t *tfx = reinterpret_cast<uint64_t *>(smem + lay.t);
    // the head's chunk arrays: shared-memory copies, or the workspace itself
    uint64_t *O = in_smem ? reinterpret_cast<uint64_t *>(smem + lay.O) : p.cpre + bhc;
    const float *ctot = in_smem ? reinterpret_cast<const float *>(smem + lay.tot) : p.ctot + bhc;
    const int *cexp = in_smem ? reinterpret_cast<const int *>(smem + lay.ce) : p.cexp + bhc;
    const float *cmx = in_smem ? reinterpret_cast<const float *>(smem + lay.cm) : p.cmax + bhc;
    int *hot = reinterpret_cast<int *>(smem + lay.hot);
    int *hv = reinterpret_cast<int *>(smem + lay.hv);
    float *hvw = reinterpret_cast<float *>(smem + lay.hvw);
    int *hist = reinterpret_cast<int *>(smem + lay.hist);
    int *idx = reinterpret_cast<int *>(smem + lay.idx);
    float *acc_s = reinterpret_cast<float *>(smem + lay.acc);
    float *qf = reinterpret_cast<float *>(smem + lay.qf);
    int *misc = reinterpret_cast<int *>(smem + lay.misc);
    uint64_t *scan64 = reinterpret_cast<uint64_t *>(misc + GM_SCAN);

    // ---- A. chunk data; the maximum score M and the largest chunk scale C
    int mk = INT_MIN, cml = INT_MIN;
    if (in_smem) {
        float *tot_s = reinterpret_cast<float *>(smem + lay.tot);
        int *ce_s = reinterpret_cast<int *>(smem + lay.ce);
        float *cm_s = reinterpret_cast<float *>(smem + lay.cm);
#pragma unroll 4
        for (int c = tid; c < nchn; c += NTH) {
            const float t = __ldcg(p.ctot + bhc + c);
            const int e = __ldcg(p.cexp + bhc + c);
            const float m = __ldcg(p.cmax + bhc + c);
            tot_s[c] = t;
            ce_s[c] = e;
            cm_s[c] = m;
            mk = max(mk, fkey(m));
            cml = max(cml, e);
        }
    } else {
        for (int c = tid; c < nchn; c += NTH) {
            mk = max(mk, fkey(__ldcg(p.cmax + bhc + c)));
            cml = max(cml, __ldcg(p.cexp + bhc + c));
        }
    }
    mk = __reduce_max_sync(FULL, mk);
    cml = __reduce_max_sync(FULL, cml);
    if (lane == 0) {
        atomicMax(misc + GM_MAX, mk);
        atomicMax(misc + GM_CMAX, cml);
    }
    team_sync<BAR, NTH>();
    const float M = fkey_inv(misc[GM_MAX]);
    const int Cm = misc[GM_CMAX];
    const float thr = M - p.tau2;  // keys with a score >= thr are re-scored

    if (tid == 0) SANTA_STAMP(TL_VALUE_ROW0 + bh, 2);
    // ---- B. fixed-point chunk totals in the global scale; hot chunks (unordered list)
    int cnt = 0;
    for (int c = tid; c < nchn; c += NTH) {
        O[c] = fixp(ctot[c], FIX_F + cexp[c] - Cm);
        cnt += cmx[c] >= thr ? 1 : 0;
    }
    cnt = __reduce_add_sync(FULL, cnt);
    if (lane == 0 && cnt) atomicAdd(misc + GM_CNT, cnt);
    team_sync<BAR, NTH>();
    int nhot = misc[GM_CNT];
    float hthr = thr;
    if (nhot > HCAP) {
        // too many qualify: keep the hottest, by a histogram of the maxima over
        // [thr, M] read from the top until HCAP would be exceeded
        for (int i = tid; i < HBINS; i += NTH) hist[i] = 0;
        team_sync<BAR, NTH>();
        const float span = fmaxf(M - thr, 1e-30f);
        for (int c = tid; c < nchn; c += NTH) {
            const float m = cmx[c];
            if (m >= thr) atomicAdd(hist + min(HBINS - 1, (int)((m - thr) / span * HBINS)), 1);
        }
        team_sync<BAR, NTH>();
        if (tid == 0) {
            int acc = 0, bin = HBINS;
            while (bin > 0 && acc + hist[bin - 1] <= HCAP) acc += hist[--bin];
            misc[GM_CNT] = bin;  // lowest bin kept (HBINS: none fits)
        }
        team_sync<BAR, NTH>();
        const int bin = misc[GM_CNT];
        hthr = bin < HBINS ? thr + span * ((float)bin / HBINS) : __int_as_float(0x7f800000);
        // (a chunk exactly on a bin edge may land in the bin below: count again)
        int cc = 0;
        for (int c = tid; c < nchn; c += NTH) cc += cmx[c] >= hthr ? 1 : 0;
        cc = __reduce_add_sync(FULL, cc);
        team_sync<BAR, NTH>();
        if (tid == 0) misc[GM_CNT] = 0;
        team_sync<BAR, NTH>();
        if (lane == 0 && cc) atomicAdd(misc + GM_CNT, cc);
        team_sync<BAR, NTH>();
        nhot = misc[GM_CNT];
        if (nhot > HCAP) nhot = 0;  // (ties at the very top: no re-scoring)
    }
    if (nhot > 0) {
        for (int c = tid; c < nchn; c += NTH)
            if (cmx[c] >= hthr) hot[atomicAdd(misc + GM_NHOT, 1)] = c;
        team_sync<BAR, NTH>();
    }

    if (tid == 0) SANTA_STAMP(TL_VALUE_ROW0 + bh, 3);
    // ---- C. heavy keys of the hot chunks: slot q = hot entry * 8 + quarter (four keys,
    // one 16-byte load); up to eight loads in flight per thread before any is acted on,
    // so HCAP hot chunks take one round.
    float *wrow = p.w + (size_t)bh * p.n_pad;
    const uint16_t *kg = p.k + ((size_t)b * p.H_kv + g) * (size_t)p.n_max * D;
    constexpr int QPC = CHUNK / 4;  // quarters per chunk
    for (int q0 = tid; q0 < nhot * QPC; q0 += 8 * NTH) {
        float4 wv[8];
        int jj[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int q = q0 + u * NTH;
            jj[u] = -1;
            wv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (q < nhot * QPC) {
                const int j = hot[q / QPC] * CHUNK + (q % QPC) * 4;
                if (j < n) {
                    jj[u] = j;
                    wv[u] = __ldcg(reinterpret_cast<const float4 *>(wrow + j));
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (jj[u] < 0) continue;
            const float wt = exp2f(thr - (float)cexp[jj[u] / CHUNK]);
            const float w4[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = jj[u] + e;
                if (j < n && w4[e] >= wt) {
                    const int pos = atomicAdd(misc + GM_NHV, 1);
                    if (pos < HKCAP) {
                        hv[pos] = j;
                        hvw[pos] = w4[e];
                    }
                }
            }
        }
    }
    team_sync<BAR, NTH>();
    const int nhv = min(misc[GM_NHV], HKCAP);

    if (tid == 0) SANTA_STAMP(TL_VALUE_ROW0 + bh, 4);
    // ---- D. re-score the heavy keys (four lanes each) and patch their chunk totals
    for (int i0 = 0; i0 < nhv; i0 += NTH / 4) {  // (every lane runs every pass: they shuffle)
        const int i = i0 + tid / 4, part = tid & 3;
        const int j = i < nhv ? hv[i] : 0;
        float shi, slo;
        rescore_key_quad<D>(kg + (size_t)j * D, qf, part, p.k2_hi, p.k2_lo, shi, slo);
        if (i < nhv && part == 0) {
            const int c = j / CHUNK;
            const int ct = cexp[c];
            const float wnew = exp2f(__fadd_rn(__fsub_rn(shi, (float)ct), slo));
            wrow[j] = wnew;
            const int e = FIX_F + ct - Cm;
            const uint64_t dx = fixp(wnew, e) - fixp(hvw[i], e);  // two's complement difference
            if (dx) atomicAdd((unsigned long long *)(O + c), (unsigned long long)dx);
        }
    }
    team_sync<BAR, NTH>();

    if (tid == 0) SANTA_STAMP(TL_VALUE_ROW0 + bh, 5);
    // ---- E. exact exclusive prefix of the G_c: a contiguous range per thread
    {
        const int per = (nchn + NTH - 1) / NTH;
        const int c0 = min(tid * per, nchn), c1 = min(c0 + per, nchn);
        uint64_t run = 0;
        for (int c = c0; c < c1; ++c) run += O[c];
        // exclusive scan of the per-thread sums over the block
        uint64_t x = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t y = __shfl_up_sync(FULL, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) scan64[warp] = x;
        team_sync<BAR, NTH>();
        if (tid == 0) {
            uint64_t a = 0;
            for (int w = 0; w < NW; ++w) {
                const uint64_t t = scan64[w];
                scan64[w] = a;
                a += t;
            }
            scan64[NW] = a;
        }
        team_sync<BAR, NTH>();
        uint64_t base = scan64[warp] + x - run;
        for (int c = c0; c < c1; ++c) {
            const uint64_t v = O[c];
            O[c] = base;
            base += v;
        }
    }
    team_sync<BAR, NTH>();
    const uint64_t Z = scan64[NW];

    if (tid == 0) SANTA_STAMP(TL_VALUE_ROW0 + bh, 6);
    // ---- F. points -> chunk (binary search on O) -> key (the chunk's 32 weights, one line)
    for (int s = tid; s < S; s += NTH) {
        const uint64_t T = __umul64hi(tfx[s], Z);
        int lo = 0, hi = nchn - 1;  // largest c with O_c <= T
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (O[mid] <= T) lo = mid; else hi = mid - 1;
        }
        const int c = lo;
        // remainder inside the chunk, in the chunk's own scale 2^-c_t (fp32)
        const float rres = __fmul_rn(__ull2float_rn(T - O[c]), exp2i(Cm - cexp[c] - FIX_F));
        const int j0 = c * CHUNK;
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
        const int pick = chunk_pick(wv, jn, rres);
        idx[s] = j0 + pick;  // (iid: overwrites this point's own uniform)
        // the V row this point selects: into L2 now, gathered in G (with one point per
        // thread; with several, the early V rows competed with the weights still to be
        // read, and the search measured slower by more than the gather gained)
        if (S <= NTH) {
            const uint16_t *vrow = p.v + (((size_t)b * p.H_kv + g) * (size_t)p.n_max + (size_t)(j0 + pick)) * D;
            prefetch_l2(vrow);
            if (D * 2 > 128) prefetch_l2(vrow + 64);
        }
    }
    team_sync<BAR, NTH>();
    if (tid == 0) SANTA_STAMP(TL_VALUE_ROW0 + bh, 7);
    // The head's weights and chunk data have been read for the last time: drop them from
    // L2 so that they are never written back (the next step's score stage rewrites them).
    l2_discard_range(wrow, (size_t)nchn * CHUNK * sizeof(float), tid, NTH);
    l2_discard_range(p.ctot + bhc, (size_t)p.nch * sizeof(float), tid, NTH);
    l2_discard_range(p.cexp + bhc, (size_t)p.nch * sizeof(int), tid, NTH);
    l2_discard_range(p.cmax + bhc, (size_t)p.nch * sizeof(float), tid, NTH);
    if (!in_smem) l2_discard_range(p.cpre + bhc, (size_t)p.nch * sizeof(uint64_t), tid, NTH);

    if (tid == 0) SANTA_STAMP(TL_VALUE_ROW0 + bh, 8);
    // ---- G. sorted indices out; each warp gathers the distinct rows of its run of
    // points (a row split between two warps is loaded by both, each with its own count)
    if (p.idx_out)
        for (int s = tid; s < S; s += NTH) p.idx_out[(size_t)bh * S + s] = idx[s];
    const uint16_t *vg = p.v + ((size_t)b * p.H_kv + g) * (size_t)p.n_max * D;
    if constexpr (G > 1 && XD) {
        {
            // The group's G heads run as one cluster (rank k = head g*G + k).  Each CTA
            // copies the G sorted lists, loads the distinct rows of its own list that no
            // lower-ranked head sampled -- so every row of the group is loaded once -- and
            // adds each, times its count in every head's list, to G partial sums.  The
            // partial sums meet in their head's CTA and are added in rank order.
            namespace cg = cooperative_groups;
            cg::cluster_group cl = cg::this_cluster();
            const int me = (int)cl.block_rank();
            int *all = reinterpret_cast<int *>(smem + lay.all);      // [G][S]: every head's list
            float *red = reinterpret_cast<float *>(smem + lay.own);  // [NW][G][D] partial sums
            float *recv = reinterpret_cast<float *>(smem + lay.recv);  // [G][D]
            // push this head's sorted list into slot `me` of every CTA of the group, once
            // every CTA is past F (the lists overlay its points and chunk arrays)
            cl.sync();
#pragma unroll
            for (int k = 0; k < G; ++k) {
                int *dst = cl.map_shared_rank(all, k) + me * S;
                for (int s = tid; s < S; s += NTH) dst[s] = idx[s];
            }
            cl.sync();  // every list is everywhere
            // each warp takes a run of points of its own list; a point leads if it is the
            // row's first occurrence here and no lower-ranked head sampled the row
            const int per = (S + NW - 1) / NW;
            const int s0 = min(warp * per, S), s1 = min(s0 + per, S);
            float acc[G][EPL];
#pragma unroll
            for (int k = 0; k < G; ++k)
#pragma unroll
                for (int e = 0; e < EPL; ++e) acc[k][e] = 0.f;
            for (int base = s0; base < s1; base += 32) {
                const int s = base + lane;
                const bool in = s < s1;
                const int j = in ? idx[s] : 0;
                bool ownr = in && (s == 0 || idx[s - 1] != j);
                int cnt[G];  // the row's count in each head's list
#pragma unroll
                for (int k = 0; k < G; ++k) {
                    cnt[k] = 0;
                    if (ownr) {
                        const int *lk = all + k * S;
                        const int lo = lower_bound_i(lk, S, j);
                        cnt[k] = (lo < S && lk[lo] == j) ? upper_bound_i(lk, S, j) - lo : 0;
                        if (k < me && cnt[k] > 0) ownr = false;  // a lower head loads it
                    }
                }
                unsigned lead = __ballot_sync(FULL, ownr);
                while (lead) {  // (lead is warp-uniform)
                    constexpr int U = G <= 4 ? 8 : 4;
                    int js[U], src[U];
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        src[u] = lead ? __ffs(lead) - 1 : 32;  // 32: no row in this slot
                        js[u] = __shfl_sync(FULL, j, src[u] & 31);
                        if (src[u] == 32) js[u] = 0;
                        lead &= lead - 1u;
                    }
                    float vv[U][EPL];
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        if constexpr (EPL == 4) {
                            const uint2 raw = *reinterpret_cast<const uint2 *>(vg + (size_t)js[u] * D + 4 * lane);
                            vv[u][0] = bf16lo_to_f32(raw.x);
                            vv[u][1] = bf16hi_to_f32(raw.x);
                            vv[u][2] = bf16lo_to_f32(raw.y);
                            vv[u][3] = bf16hi_to_f32(raw.y);
                        } else {
                            const uint32_t raw = *reinterpret_cast<const uint32_t *>(vg + (size_t)js[u] * D + 2 * lane);
                            vv[u][0] = bf16lo_to_f32(raw);
                            vv[u][1] = bf16hi_to_f32(raw);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < U; ++u)
#pragma unroll
                        for (int k = 0; k < G; ++k) {
                            const int c = __shfl_sync(FULL, cnt[k], src[u] & 31);
                            const float cf = src[u] < 32 ? (float)c : 0.f;
#pragma unroll
                            for (int e = 0; e < EPL; ++e) acc[k][e] = __fmaf_rn(cf, vv[u][e], acc[k][e]);
                        }
                }
            }
            // partial sums of this CTA for each head (over the lists: once every warp is past
            // them) -> slot `me` of that head's CTA
            team_sync<BAR, NTH>();
#pragma unroll
            for (int k = 0; k < G; ++k)
#pragma unroll
                for (int e = 0; e < EPL; ++e) red[(warp * G + k) * D + EPL * lane + e] = acc[k][e];
            team_sync<BAR, NTH>();
            for (int i = tid; i < G * D; i += NTH) {
                const int k = i / D, dd = i % D;
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < NW; ++w) sum = __fadd_rn(sum, red[(w * G + k) * D + dd]);
                cl.map_shared_rank(recv, k)[me * D + dd] = sum;
            }
            cl.sync();  // every partial sum has arrived
            for (int i = tid; i < D; i += NTH) {
                float sum = 0.f;
#pragma unroll
                for (int jj = 0; jj < G; ++jj) sum = __fadd_rn(sum, recv[jj * D + i]);
                store_out(p, (size_t)bh * D + i, __fdiv_rn(sum, (float)S));
            }
            if (tid == 0) SANTA_STAMP(TL_VALUE_ROW0 + bh, 10);
            return;
        }
    }
    // distinct rows of this head's sorted list (first occurrences, in order) ...
    int *lead = reinterpret_cast<int *>(smem + lay.lead);
    {
        const int per = (S + NTH - 1) / NTH;
        const int s0 = min(tid * per, S), s1 = min(s0 + per, S);
        int cnt = 0;
        for (int s = s0; s < s1; ++s) cnt += (s == 0 || idx[s] != idx[s - 1]) ? 1 : 0;
        int nlead;
        int pos = team_excl_scan<BAR, NTH>(cnt, tid, misc, &nlead);
        for (int s = s0; s < s1; ++s)
            if (s == 0 || idx[s] != idx[s - 1]) lead[pos++] = s;
        if (tid == 0) lead[nlead] = S;
        team_sync<BAR, NTH>();
        // ... then each thread loads 16-byte pieces (8 dimensions) of every RSTEP-th
        // distinct row, eight loads in flight, and adds them times their counts; the
        // RSTEP partial sums of each piece are added in a fixed order
        constexpr int NPC = D * 2 / 16;   // 16-byte pieces per row
        constexpr int RSTEP = NTH / NPC;   // rows in parallel
        const int piece = tid % NPC, r0 = tid / NPC;
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
        for (int l0 = r0; l0 < nlead; l0 += 8 * RSTEP) {
            uint4 raw[8];
            float cf[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int li = l0 + u * RSTEP;
                cf[u] = 0.f;
                raw[u] = make_uint4(0u, 0u, 0u, 0u);
                if (li < nlead) {
                    const int s = lead[li];
                    cf[u] = (float)(lead[li + 1] - s);
                    raw[u] = *reinterpret_cast<const uint4 *>(vg + (size_t)idx[s] * D + 8 * piece);
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t wv[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[2 * i] = __fmaf_rn(cf[u], bf16lo_to_f32(wv[i]), acc[2 * i]);
                    acc[2 * i + 1] = __fmaf_rn(cf[u], bf16hi_to_f32(wv[i]), acc[2 * i + 1]);
                }
            }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) acc_s[(r0 * NPC + piece) * 8 + e] = acc[e];
        team_sync<BAR, NTH>();
        if (tid == 0) SANTA_STAMP(TL_VALUE_ROW0 + bh, 9);
        for (int i = tid; i < D; i += NTH) {
            float sum = 0.f;
            for (int r = 0; r < RSTEP; ++r) sum = __fadd_rn(sum, acc_s[(r * NPC + i / 8) * 8 + i % 8]);
            store_out(p, (size_t)bh * D + i, __fdiv_rn(sum, (float)S));
        }
    }
    if (tid == 0) SANTA_STAMP(TL_VALUE_ROW0 + bh, 10);
}

// One CTA per (b, h_q), a programmatic dependent of the score kernel (four CTAs per SM:
// all B*H_q CTAs of a B=16, H_q=32 step fit in one wave).  With SANTA_GROUP_DEDUP the host
// launches the G heads of a group as one cluster.
// VAR: GATHER_XD (group dedup, launched as clusters of G; G > 1) and GATHER_IID (i.i.d.
// points) select the paths at compile time, so that each launch carries only the code it
// runs (the value stage runs each phase once per CTA: fetching a larger kernel's
// instructions measured about 4 us slower at B=16).
template <int D, int G, int VAR, int NTH = (VAR & GATHER_WIDE) ? NT_WIDE : NT>
__global__ void __launch_bounds__(NTH, NTH == NT ? 4 : 1) santa_gather_kernel(const Params p)
{
    constexpr bool XD = (VAR & GATHER_XD) != 0 && G > 1, IID = (VAR & GATHER_IID) != 0;
    static_assert(!(XD && NTH != NT), "group dedup runs with the narrow team");
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, bh = blockIdx.x;
    if (tid == 0) SANTA_STAMP(TL_VALUE_ROW0 + bh, 0);
    const int n = value_len(p, bh / p.H_q);
    if (n == 0) {  // (every CTA of a cluster shares b, so all of them leave here)
        value_empty<D, NTH>(p, bh, tid);
        return;
    }
    const GatherSmem lay = gather_smem(D, G, p.S, p.nch, p.mode, XD, NTH);
    value_prologue<D, G, NTH, 0, IID>(p, bh, smem, lay, tid);
    pdl_wait();  // the score kernel's results are complete and visible from here on
    __syncthreads();
    if (tid == 0) SANTA_STAMP(TL_VALUE_ROW0 + bh, 1);
    value_main<D, G, NTH, 0, XD>(p, bh, n, smem, lay, tid);
}

}  // namespace santa
