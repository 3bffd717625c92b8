// santa_sample.cuh -- the fused SANTA decode kernel (sampled value stage), sm_103a.
//
// "Stochastic Sparse Attention for Memory-Bound Inference" (abstract): the score stage
// reads all n_k keys and forms the post-softmax distribution; the value stage samples
// S << n_k indices from it (stratified or systematic sampling) and gather-adds only
// those V rows, scaled by 1/S.
//
// One persistent kernel does the whole step.  Work items are splits (b, g, r): L
// consecutive keys of KV head g of batch row b.  CTAs take items from an atomic counter
// and stream the items' K rows as 16 KB tiles through a 4-stage ring filled by 1-D TMA
// bulk copies.  Per tile and per key the warp computes the G query heads' scores with
// packed fp32 FMAs (each K element read from shared memory once, used G times).  Scores
// within a window of the running maximum are recomputed with an error-free double-float
// dot product, because the heaviest keys' rounding errors shift every later CDF
// boundary.  At the end of a split the CTA writes, per query head, the fp32 weights
// w_j = 2^(s_j log2 e - c_r) (c_r an integer near the split maximum), the exact fp64
// prefix of 32-key chunk totals, and the split total.  The CTA that completes the last
// split of a group (b, g) merges the split totals exactly (the split scales are powers
// of two), draws the S sorted points of each query head, finds their keys by a
// split -> chunk -> key search, and gather-adds each distinct V row once for all G heads
// of the group.
#pragma once

#include "santa_common.cuh"

namespace santa {

template <int D, int G>
struct SampleCfg {
    static constexpr int P = D / 16;            // lanes per key in the score loop
    static constexpr int KW = 64 / P;           // keys per warp and tile (2 per lane group)
    static constexpr int TK = NWARP * KW;       // keys per tile
    static constexpr int ROWB = 2 * D;          // bytes per K row
    static constexpr int NSTAGE = 4;
    static constexpr int V = 2 * G;             // partial dots per lane
    static constexpr int NV = V >= P ? V / P : 1;   // scores per lane after the reduction
    static constexpr int REP = V >= P ? 1 : P / V;  // lanes holding the same score
    static constexpr int EPL = D / 32;          // V elements per lane in the gather
    static_assert(TK * ROWB == TILE_BYTES, "tile size");
    static_assert(LMIN % TK == 0, "split length must be a multiple of the tile");

    __host__ __device__ static constexpr int vidx(int sub, int i) { return V >= P ? sub * NV + i : sub / REP; }
    __host__ __device__ static constexpr int head_of(int lane, int i) { return vidx(lane % P, i) % G; }
    __host__ __device__ static constexpr int key2_of(int lane, int i) { return vidx(lane % P, i) / G; }
    // Flipping lane bit m leaves the heads of every score slot unchanged.
    __host__ __device__ static constexpr bool same_heads(int m)
    {
        for (int l = 0; l < 32; ++l)
            for (int i = 0; i < NV; ++i)
                if (head_of(l ^ m, i) != head_of(l, i)) return false;
        return true;
    }
};

// Shared-memory carve-up of the sampled kernel (host and device agree on it).
struct SampleSmem {
    int stage, bar, desc, qf, tmax, misc, nb, prefix, ctot, region, total;
};

__host__ __device__ inline int next_pow2(int x)
{
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

__host__ __device__ inline SampleSmem sample_smem(int D, int G, int B, int S, int ns_max_used, int mode)
{
    SampleSmem s{};
    int off = 0;
    s.stage = off; off += 4 * TILE_BYTES;
    s.bar = off; off += 4 * 8;
    s.desc = off; off += 4 * 16;
    s.qf = off; off += G * D * 4;
    s.tmax = off; off += NWARP * G * 4;
    s.misc = off; off += 16 * 4;
    s.nb = off; off += (int)align_up((size_t)B * 4, 16);
    s.prefix = off; off += (int)align_up((size_t)(B + 1) * 4, 16);
    s.ctot = off; off += (int)align_up((size_t)NWARP * G * 4, 16) + G * (LMAX / CHUNK) * 8;
    off = (int)align_up((size_t)off, 128);
    s.region = off;
    const int score_bytes = 2 * G * LMAX * 4;
    const int Sp = (mode == MODE_IID) ? next_pow2(S) : S;
    const int idx_bytes = (int)align_up((size_t)G * Sp * 4, 16);
    const int phaseA = (int)align_up((size_t)G * ns_max_used * 4, 16) + G * (ns_max_used + 1) * 8 + 64;
    const int phaseC = (int)align_up((size_t)G * S * 4, 16) + (int)align_up((size_t)G * S * G * 2, 16) +
                       NWARP * G * D * 4 + 64;
    int ep = idx_bytes + (phaseA > phaseC ? phaseA : phaseC);
    off += score_bytes > ep ? score_bytes : ep;
    s.total = off;
    return s;
}

// Descriptor of a staged tile.
enum : int { DESC_END = -1 };
enum : int { FLAG_LAST = 1, FLAG_ZERO = 2 };

struct Item {
    int b, g, r, n, ns;
};

__device__ __forceinline__ Item decode_item(int it, const int *prefix, const int *nb, int B, int H_kv, int L)
{
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= it) lo = mid; else hi = mid - 1;
    }
    Item x;
    x.b = lo;
    x.n = nb[lo];
    x.ns = x.n > 0 ? (x.n + L - 1) / L : 1;
    const int local = it - prefix[lo];
    x.g = local / x.ns;
    x.r = local % x.ns;
    (void)H_kv;
    return x;
}

// Reduce-scatter of the V partial dots of a lane group of P lanes: after it the lane
// keeps the sums of the value slots given by SampleCfg::vidx.
template <int M, int C, int V>
__device__ __forceinline__ void rs_step(float (&val)[V], int sub)
{
    if constexpr (M >= 1) {
        if constexpr (C > 1) {
            constexpr int H = C / 2;
            const bool up = (sub & M) != 0;
#pragma unroll
            for (int i = 0; i < H; ++i) {
                const float send = up ? val[i] : val[i + H];
                const float recv = __shfl_xor_sync(0xffffffffu, send, M);
                val[i] = __fadd_rn(up ? val[i + H] : val[i], recv);
            }
            rs_step<M / 2, H, V>(val, sub);
        } else {
            val[0] = __fadd_rn(val[0], __shfl_xor_sync(0xffffffffu, val[0], M));
            rs_step<M / 2, 1, V>(val, sub);
        }
    }
}

// fp32 dots of 2 keys (rows kbase, kbase+1 of the tile) with the G query heads; lane
// sub of the group holds 16 elements: 16-byte chunks sub and sub + P of each row.
template <int D, int G>
__device__ __forceinline__ void tile_dots(const uint8_t *tile, int kbase, int sub,
                                          const unsigned long long (&qp)[G][8], float (&val)[2 * G])
{
    using C = SampleCfg<D, G>;
    unsigned long long acc[2][G];
#pragma unroll
    for (int kk = 0; kk < 2; ++kk)
#pragma unroll
        for (int h = 0; h < G; ++h) acc[kk][h] = 0ull;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
        const uint8_t *row = tile + (kbase + kk) * C::ROWB;
        const uint4 a = *reinterpret_cast<const uint4 *>(row + 16 * sub);
        const uint4 c = *reinterpret_cast<const uint4 *>(row + 16 * (sub + C::P));
        const uint32_t wv[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const unsigned long long kp = bf16x2_to_f32x2(wv[i]);
#pragma unroll
            for (int h = 0; h < G; ++h) ffma2(acc[kk][h], qp[h][i], kp);
        }
    }
#pragma unroll
    for (int kk = 0; kk < 2; ++kk)
#pragma unroll
        for (int h = 0; h < G; ++h) val[kk * G + h] = f32x2_sum(acc[kk][h]);
    rs_step<C::P / 2, 2 * G, 2 * G>(val, sub);
}

// Error-free dot of one staged K row with query head qf_h (fp32 copies of bf16 values),
// by the whole warp; returns the score in log2 units as a normalised pair (hi, lo).
template <int D>
__device__ __forceinline__ void refine_score(const uint8_t *row, const float *qf_h, int lane, float k2_hi,
                                             float k2_lo, float &hi, float &lo)
{
    float s, e, t;
    if constexpr (D == 128) {
        const uint2 kw = *reinterpret_cast<const uint2 *>(row + 8 * lane);
        const float4 qv = *reinterpret_cast<const float4 *>(qf_h + 4 * lane);
        const float p0 = __fmul_rn(qv.x, bf16lo_to_f32(kw.x));
        const float p1 = __fmul_rn(qv.y, bf16hi_to_f32(kw.x));
        const float p2 = __fmul_rn(qv.z, bf16lo_to_f32(kw.y));
        const float p3 = __fmul_rn(qv.w, bf16hi_to_f32(kw.y));
        two_sum(p0, p1, s, e);
        two_sum(s, p2, s, t);
        e = __fadd_rn(e, t);
        two_sum(s, p3, s, t);
        e = __fadd_rn(e, t);
    } else {
        const uint32_t kw = *reinterpret_cast<const uint32_t *>(row + 4 * lane);
        const float2 qv = *reinterpret_cast<const float2 *>(qf_h + 2 * lane);
        two_sum(__fmul_rn(qv.x, bf16lo_to_f32(kw)), __fmul_rn(qv.y, bf16hi_to_f32(kw)), s, e);
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
        const float s2 = __shfl_xor_sync(0xffffffffu, s, m);
        const float e2 = __shfl_xor_sync(0xffffffffu, e, m);
        two_sum(s, s2, s, t);
        e = __fadd_rn(__fadd_rn(e, e2), t);
    }
    fast_two_sum(s, e, s, e);
    // (s + e) * (k2_hi + k2_lo) to about 2^-46 relative
    const float P = __fmul_rn(s, k2_hi);
    float E = __fmaf_rn(s, k2_hi, -P);
    E = __fmaf_rn(s, k2_lo, E);
    E = __fmaf_rn(e, k2_hi, E);
    fast_two_sum(P, E, hi, lo);
}

// ------------------------------------------------------------------ block helpers

// Exclusive block scan of one int per thread; returns the block total via *total.
__device__ __forceinline__ int block_excl_scan(int v, int *scratch /*NWARP+1 ints*/, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int w = 0; w < NWARP; ++w) {
            const int t = scratch[w];
            scratch[w] = acc;
            acc += t;
        }
        scratch[NWARP] = acc;
    }
    __syncthreads();
    const int res = scratch[warp] + x - v;
    *total = scratch[NWARP];
    __syncthreads();
    return res;
}

__device__ __forceinline__ int lower_bound_i(const int *a, int n, int key)
{
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] < key) lo = mid + 1; else hi = mid;
    }
    return lo;
}

__device__ __forceinline__ int upper_bound_i(const int *a, int n, int key)
{
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] <= key) lo = mid + 1; else hi = mid;
    }
    return lo;
}


// ------------------------------------------------------------------ the kernel

// misc[] words of the sampled kernel's shared block
enum : int { MISC_SCAN = 0 /* NWARP+1 words */, MISC_LAST = 12 };

template <int D, int G>
__global__ void __launch_bounds__(NT, (G <= 4 ? 2 : 1)) santa_sample_kernel(const Params p)
{
    using C = SampleCfg<D, G>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sub = lane % C::P, grp = lane / C::P;
    const int B = p.B, H_kv = p.H_kv, H_q = p.H_q, L = p.L;
    const int ns_used = (p.n_max + L - 1) / L;
    const SampleSmem lay = sample_smem(D, G, B, p.S, ns_used, p.mode);

    uint8_t *stage = smem + lay.stage;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + lay.bar);
    int4 *sdesc = reinterpret_cast<int4 *>(smem + lay.desc);
    float *qf = reinterpret_cast<float *>(smem + lay.qf);
    float *tmax = reinterpret_cast<float *>(smem + lay.tmax);
    int *misc = reinterpret_cast<int *>(smem + lay.misc);
    int *nb = reinterpret_cast<int *>(smem + lay.nb);
    int *prefix = reinterpret_cast<int *>(smem + lay.prefix);
    float *red = reinterpret_cast<float *>(smem + lay.ctot);
    double *ctot = reinterpret_cast<double *>(smem + lay.ctot + align_up((size_t)NWARP * G * 4, 16));
    uint8_t *region = smem + lay.region;
    float *sc_hi = reinterpret_cast<float *>(region);
    float *sc_lo = sc_hi + G * LMAX;
    const float NEG_INF = __int_as_float(0xff800000);

    // ---- item space: per batch row, H_kv * ceil(n_b / L) splits (H_kv zero items if n_b = 0)
    {
        constexpr int PER = (BMAX + NT - 1) / NT;
        int cnt[PER];
        int local = 0;
        bool bad = false;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int b = tid * PER + i;
            cnt[i] = 0;
            if (b < B) {
                int n = p.seq_lens[b];
                if (n < 0 || n > p.n_max) {
                    bad = true;
                    n = 0;
                }
                nb[b] = n;
                cnt[i] = H_kv * (n > 0 ? (n + L - 1) / L : 1);
                local += cnt[i];
            }
        }
        if (bad && blockIdx.x == 0) set_dev_error(p.ctrl, DEV_BAD_SEQLEN);
        int total;
        int run = block_excl_scan(local, misc + MISC_SCAN, &total);
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int b = tid * PER + i;
            if (b < B) prefix[b] = run;
            run += cnt[i];
        }
        if (tid == 0) prefix[B] = total;
    }
    if (tid == 0) {
        for (int s = 0; s < C::NSTAGE; ++s) mbar_init(&bars[s], 1);
        mbar_fence_init();
    }
    __syncthreads();
    const int total_items = prefix[B];

    // ---- producer (thread 0): the stream of tiles of the items it takes, in order
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
        mbar_arrive_tx(&bars[slot], bytes);
        bulk_g2s(stage + slot * TILE_BYTES, p.k + (pr_row0 + (long long)pr_tile * C::TK) * D, bytes, &bars[slot],
                 policy);
        ++pr_tile;
    };
    if (tid == 0)
        for (int s = 0; s < C::NSTAGE; ++s) produce(s);

    // ---- consumers (all threads; control flow is uniform across the CTA)
    unsigned long long qp[G][8];
    float runmax[G];
#pragma unroll
    for (int h = 0; h < G; ++h) runmax[h] = NEG_INF;
    Item cur{0, 0, 0, 0, 1};
    int valid = 0;
    bool aborted = false;
    int it = 0;

    for (;; ++it) {
        const int slot = it % C::NSTAGE;
        const uint32_t par = (uint32_t)(it / C::NSTAGE) & 1u;
        const bool ok = mbar_wait_bounded(&bars[slot], par, p.wait_ns);
        if (__syncthreads_or(!ok)) {
            aborted = true;
            break;
        }
        // everyone is done with the previous tile: refill its slot, fold its maxima in
        if (tid == 0 && it > 0) produce((it - 1) % C::NSTAGE);
        if (it > 0) {
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int w = 0; w < NWARP; ++w) runmax[h] = fmaxf(runmax[h], tmax[w * G + h]);
        }
        const int4 dsc = sdesc[slot];
        if (dsc.x == DESC_END) break;

        if (dsc.w & FLAG_ZERO) {
            // empty sequence: out = 0 and idx = -1 for the group's G query heads
            const Item x = decode_item(dsc.x, prefix, nb, B, H_kv, L);
            for (int i = tid; i < G * D; i += NT) p.out[((size_t)x.b * H_q + x.g * G) * D + i] = 0.f;
            if (p.idx_out)
                for (int i = tid; i < G * p.S; i += NT) p.idx_out[((size_t)x.b * H_q + x.g * G) * p.S + i] = -1;
#pragma unroll
            for (int h = 0; h < G; ++h) runmax[h] = NEG_INF;
            if (lane == 0)
                for (int h = 0; h < G; ++h) tmax[warp * G + h] = NEG_INF;
            continue;
        }

        const int tile = dsc.y, rows = dsc.z;
        if (tile == 0) {
            cur = decode_item(dsc.x, prefix, nb, B, H_kv, L);
            valid = min(L, cur.n - cur.r * L);
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
                sc_hi[h * LMAX + tile * C::TK + key] = s2[i];
                sc_lo[h * LMAX + tile * C::TK + key] = 0.f;
            }
        }
        // warp maximum of this tile per head (lanes that share heads)
        float wm[C::NV];
#pragma unroll
        for (int i = 0; i < C::NV; ++i) wm[i] = s2[i];
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            if (C::same_heads(m)) {
#pragma unroll
                for (int i = 0; i < C::NV; ++i) wm[i] = fmaxf(wm[i], __shfl_xor_sync(0xffffffffu, wm[i], m));
            }
        }
        // recompute, error-free, the scores within tau2 of the running maximum
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
                    sc_hi[hh * LMAX + tile * C::TK + key] = hi;
                    sc_lo[hh * LMAX + tile * C::TK + key] = lo;
                }
            }
        }
        // publish the warp maxima per head (one lane per class of lanes sharing heads)
        {
            bool first = true;
#pragma unroll
            for (int m = 1; m < 32; m <<= 1)
                if (C::same_heads(m) && (lane & m)) first = false;
            if (first) {
#pragma unroll
                for (int i = 0; i < C::NV; ++i) tmax[warp * G + C::head_of(lane, i)] = wm[i];
            }
        }

        if (!(dsc.w & FLAG_LAST)) continue;

        // ================= end of split (b, g, r): weights, chunk prefix, split total
        __syncthreads();
        const int b = cur.b, g = cur.g, r = cur.r;
        const int nchunks = (valid + CHUNK - 1) / CHUNK;
        {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float mx = NEG_INF;
                for (int j = tid; j < valid; j += NT) mx = fmaxf(mx, sc_hi[h * LMAX + j]);
#pragma unroll
                for (int m = 16; m >= 1; m >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
                if (lane == 0) red[warp * G + h] = mx;
            }
        }
        __syncthreads();
        int cr[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float m = NEG_INF;
#pragma unroll
            for (int w = 0; w < NWARP; ++w) m = fmaxf(m, red[w * G + h]);
            m = fminf(fmaxf(m, -16777216.f), 16777216.f);
            cr[h] = (int)ceilf(m);
        }
        // weights w_j = 2^(s_j - c_r); a warp task covers 4 chunks of one head, 4 keys a lane
        {
            const int cg = (nchunks + 3) / 4;
            for (int task = warp; task < G * cg; task += NWARP) {
                const int h = task / cg, c4 = task % cg;
                const int chunk = c4 * 4 + lane / 8;
                const int j0 = chunk * CHUNK + (lane % 8) * 4;
                int crh = cr[0];
#pragma unroll
                for (int hh = 1; hh < G; ++hh) crh = (h == hh) ? cr[hh] : crh;
                const float cf = (float)crh;
                float wq[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int j = j0 + u;
                    wq[u] = 0.f;
                    if (j < valid) {
                        const float dd = __fadd_rn(__fsub_rn(sc_hi[h * LMAX + j], cf), sc_lo[h * LMAX + j]);
                        wq[u] = exp2f(dd);
                    }
                }
                if (chunk < nchunks) {
                    float *wdst = p.w + ((size_t)b * H_q + g * G + h) * p.n_pad + (size_t)r * L + j0;
                    *reinterpret_cast<float4 *>(wdst) = make_float4(wq[0], wq[1], wq[2], wq[3]);
                }
                float s, e, t;
                two_sum(wq[0], wq[1], s, e);
                two_sum(s, wq[2], s, t);
                e = __fadd_rn(e, t);
                two_sum(s, wq[3], s, t);
                e = __fadd_rn(e, t);
#pragma unroll
                for (int m = 4; m >= 1; m >>= 1) {
                    const float s_ = __shfl_xor_sync(0xffffffffu, s, m);
                    const float e_ = __shfl_xor_sync(0xffffffffu, e, m);
                    two_sum(s, s_, s, t);
                    e = __fadd_rn(__fadd_rn(e, e_), t);
                }
                if ((lane % 8) == 0 && chunk < nchunks)
                    ctot[h * (LMAX / CHUNK) + chunk] = __dadd_rn((double)s, (double)e);
            }
        }
        __syncthreads();
        // exclusive fp64 prefix of the chunk totals; split total and scale
        if (warp < G) {
            const int h = warp;
            const double x = lane < nchunks ? ctot[h * (LMAX / CHUNK) + lane] : 0.0;
            double incl = x;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl = __dadd_rn(incl, y);
            }
            const size_t bh = (size_t)b * H_q + g * G + h;
            if (lane < nchunks) p.coff[bh * p.nch + (size_t)r * (L / CHUNK) + lane] = __dsub_rn(incl, x);
            const double tot = __shfl_sync(0xffffffffu, incl, 31);
            int crh = cr[0];
#pragma unroll
            for (int hh = 1; hh < G; ++hh) crh = (h == hh) ? cr[hh] : crh;
            if (lane == 0) {
                p.split_W[bh * p.ns_max + r] = tot;
                p.split_c[bh * p.ns_max + r] = crh;
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

        // ================= group epilogue: every split of (b, g) is done
        const int n = cur.n, ns = cur.ns, S = p.S;
        const int Sp = (p.mode == MODE_IID) ? next_pow2(S) : S;
        int *ep_idx = reinterpret_cast<int *>(region);
        uint8_t *ep_rest = region + align_up((size_t)G * Sp * 4, 16);
        int *ep_c = reinterpret_cast<int *>(ep_rest);
        double *ep_O = reinterpret_cast<double *>(ep_rest + align_up((size_t)G * ns * 4, 16));
        int *ep_C = reinterpret_cast<int *>(ep_O + G * (ns + 1));
        const size_t bh0 = (size_t)b * H_q + g * G;

        for (int i = tid; i < G * ns; i += NT) {
            const int h = i / ns, rr = i % ns;
            ep_c[i] = __ldcg(p.split_c + (bh0 + h) * p.ns_max + rr);
            ep_O[h * (ns + 1) + rr] = __ldcg(p.split_W + (bh0 + h) * p.ns_max + rr);
        }
        __syncthreads();
        if (warp < G) {
            // split offsets O_r = sum_{r' < r} W_r' 2^(c_r' - C), exact scaling, fp64 sums
            const int h = warp;
            int cm = INT_MIN;
            for (int rr = lane; rr < ns; rr += 32) cm = max(cm, ep_c[h * ns + rr]);
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) cm = max(cm, __shfl_xor_sync(0xffffffffu, cm, m));
            double carry = 0.0;
            for (int base = 0; base < ns; base += 32) {
                const int rr = base + lane;
                double x = 0.0;
                if (rr < ns) x = __dmul_rn(ep_O[h * (ns + 1) + rr], pow2d(ep_c[h * ns + rr] - cm));
                double incl = x;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const double y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl = __dadd_rn(incl, y);
                }
                __syncwarp();
                if (rr < ns) ep_O[h * (ns + 1) + rr] = __dadd_rn(carry, __dsub_rn(incl, x));
                carry = __dadd_rn(carry, __shfl_sync(0xffffffffu, incl, 31));
            }
            if (lane == 0) {
                ep_O[h * (ns + 1) + ns] = carry;  // Z in the group scale 2^-C
                ep_C[h] = cm;
            }
        }
        // iid: the S uniforms of each head, sorted (bitonic, keys are the 32-bit draws)
        if (p.mode == MODE_IID) {
            unsigned *ukeys = reinterpret_cast<unsigned *>(ep_idx);
            for (int i = tid; i < G * Sp; i += NT) {
                const int h = i / Sp, s = i % Sp;
                unsigned u = 0xffffffffu;
                if (s < S) {
                    uint64_t rnd[4];
                    philox_block(p.seed, (uint64_t)(s / 4), b, g * G + h, 3, rnd);
                    u = (unsigned)(rnd[s % 4] >> 32);
                }
                ukeys[i] = u;
            }
            __syncthreads();
            for (int kk = 2; kk <= Sp; kk <<= 1) {
                for (int jj = kk >> 1; jj > 0; jj >>= 1) {
                    for (int i = tid; i < G * Sp; i += NT) {
                        const int h = i / Sp, s = i % Sp;
                        const int partner = s ^ jj;
                        if (partner > s) {
                            unsigned *a = ukeys + h * Sp;
                            const bool asc = (s & kk) == 0;
                            const unsigned x = a[s], y = a[partner];
                            if ((x > y) == asc) {
                                a[s] = y;
                                a[partner] = x;
                            }
                        }
                    }
                    __syncthreads();
                }
            }
        }
        __syncthreads();

        // ---- points -> split (O, smem) -> chunk (coff) -> key (w): i = min{j : C_j > t}
        for (int pi = tid; pi < G * S; pi += NT) {
            const int h = pi / S, s = pi % S;
            double t;
            if (p.mode != MODE_IID) {
                t = sample_point(p.mode, p.seed, b, g * G + h, s, p.rS);
            } else {
                const unsigned u = reinterpret_cast<const unsigned *>(ep_idx)[h * Sp + s];
                t = __dmul_rn(__uint2double_rn(u), 0x1p-32);
            }
            const double *O = ep_O + h * (ns + 1);
            const double T = __dmul_rn(t, O[ns]);
            const uint64_t Tk = dkey(T);
            int lo = 0, hi = ns - 1;  // largest r with O_r <= T
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (dkey(O[mid]) <= Tk) lo = mid; else hi = mid - 1;
            }
            const int rr = lo;
            const double Tl = __dmul_rn(__dsub_rn(T, O[rr]), pow2pos(ep_C[h] - ep_c[h * ns + rr]));
            const int vr = min(L, n - rr * L);
            const int ncr = (vr + CHUNK - 1) / CHUNK;
            const double *cof = p.coff + (bh0 + h) * p.nch + (size_t)rr * (L / CHUNK);
            const uint64_t Tlk = dkey(Tl);
            int clo = 0, chi = ncr - 1;  // largest chunk with offset <= Tl
            while (clo < chi) {
                const int mid = (clo + chi + 1) >> 1;
                if (dkey(__ldcg(cof + mid)) <= Tlk) clo = mid; else chi = mid - 1;
            }
            const float rres = (float)__dsub_rn(Tl, __ldcg(cof + clo));
            const int j0 = rr * L + clo * CHUNK;
            const int jend = min(j0 + CHUNK, n);
            const float *wrow = p.w + (bh0 + h) * p.n_pad;
            float acc = 0.f;
            int pick = -1, lastpos = j0;
            for (int j = j0; j < jend; ++j) {
                const float wj = __ldcg(wrow + j);
                if (wj > 0.f) lastpos = j;
                acc = __fadd_rn(acc, wj);
                if (acc > rres) {
                    pick = j;
                    break;
                }
            }
            if (pick < 0) pick = lastpos;  // only when rounding put t past the chunk's mass
            ep_idx[h * Sp + s] = pick;     // (iid: overwrites this point's own uniform)
            if (p.idx_out) p.idx_out[(bh0 + h) * S + s] = pick;
        }
        __syncthreads();

        // ---- gather-add: each distinct V row of the group loaded once, weighted per head
        {
            int *ep_lead = reinterpret_cast<int *>(ep_rest);
            uint16_t *ep_cnt = reinterpret_cast<uint16_t *>(ep_rest + align_up((size_t)G * S * 4, 16));
            float *ep_acc = reinterpret_cast<float *>(ep_rest + align_up((size_t)G * S * 4, 16) +
                                                      align_up((size_t)G * S * G * 2, 16));
            const int total = G * S;
            const int per = (total + NT - 1) / NT;
            const int e0 = min(tid * per, total), e1 = min(e0 + per, total);
            auto is_lead = [&](int e) {
                const int h = e / S, s = e % S;
                const int j = ep_idx[h * Sp + s];
                bool lead = (s == 0) || ep_idx[h * Sp + s - 1] != j;
                for (int h2 = 0; h2 < h && lead; ++h2) {
                    const int q2 = lower_bound_i(ep_idx + h2 * Sp, S, j);
                    if (q2 < S && ep_idx[h2 * Sp + q2] == j) lead = false;
                }
                return lead;
            };
            int cnt = 0;
            for (int e = e0; e < e1; ++e) cnt += is_lead(e) ? 1 : 0;
            int nlead;
            int pos = block_excl_scan(cnt, misc + MISC_SCAN, &nlead);
            for (int e = e0; e < e1; ++e) {
                if (!is_lead(e)) continue;
                const int j = ep_idx[(e / S) * Sp + e % S];
                ep_lead[pos] = j;
#pragma unroll
                for (int h = 0; h < G; ++h)
                    ep_cnt[pos * G + h] = (uint16_t)(upper_bound_i(ep_idx + h * Sp, S, j) -
                                                     lower_bound_i(ep_idx + h * Sp, S, j));
                ++pos;
            }
            __syncthreads();
            float acc[G][C::EPL];
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < C::EPL; ++e) acc[h][e] = 0.f;
            const uint16_t *vg = p.v + ((size_t)b * H_kv + g) * (size_t)p.n_max * D;
            constexpr int U = 4;
            for (int l0 = warp * U; l0 < nlead; l0 += NWARP * U) {
                float vv[U][C::EPL];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int li = l0 + u;
                    const int j = li < nlead ? ep_lead[li] : 0;
                    if constexpr (C::EPL == 4) {
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
                    if (li >= nlead) break;
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const float cf = (float)ep_cnt[li * G + h];
#pragma unroll
                        for (int e = 0; e < C::EPL; ++e) acc[h][e] = __fmaf_rn(cf, vv[u][e], acc[h][e]);
                    }
                }
            }
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < C::EPL; ++e) ep_acc[(warp * G + h) * D + C::EPL * lane + e] = acc[h][e];
            __syncthreads();
            for (int i = tid; i < G * D; i += NT) {
                float s = 0.f;
#pragma unroll
                for (int w = 0; w < NWARP; ++w) s = __fadd_rn(s, ep_acc[w * G * D + i]);
                p.out[bh0 * D + i] = __fdiv_rn(s, (float)S);
            }
        }
        if (tid == 0) p.ctrl[CTRL_GROUPS + b * H_kv + g] = 0;
        __syncthreads();
    }

    if (aborted) {
        // give the copies still in flight a bounded chance to land before the CTA exits
        if (tid == 0) {
            set_dev_error(p.ctrl, DEV_TIMEOUT);
            for (int k = 0; k < C::NSTAGE - 1; ++k) {
                const int j = it + k;
                mbar_wait_bounded(&bars[j % C::NSTAGE], (uint32_t)(j / C::NSTAGE) & 1u, p.wait_ns);
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
