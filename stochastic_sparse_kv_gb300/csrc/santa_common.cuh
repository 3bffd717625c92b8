// santa_common.cuh -- device helpers, constants and launch parameters shared by the
// SANTA kernels.
//
// Everything here serves the kernels of libsanta.so: the sampled path (a streaming
// score kernel that leaves softmax weights and CDF pieces in the workspace, then a
// value-stage kernel that draws stratified/systematic points, searches the CDF and
// gather-adds V rows; "Stochastic Sparse Attention for Memory-Bound Inference",
// abstract) and the dense split-K baseline.  sm_103a only.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace santa {

constexpr int NT = 256;              // threads per CTA
constexpr int NWARP = NT / 32;       // 8 warps
constexpr int DENSE_UNIT = 512;      // keys per work unit (and per partial) of the dense kernel
constexpr int CHUNK = 32;            // keys per CDF chunk (one 128-byte line of fp32 w)
constexpr int NS_LIMIT = 1024;       // most dense splits one sequence may have
constexpr int NMAX_LIMIT = 524288;   // longest KV cache (keys)
constexpr int BMAX = 1024;           // batch rows per call
constexpr int SMAX = 4096;           // samples per (b, h)

// Control block (int32 words at the start of the workspace).
enum : int { CTRL_ERR = 0, CTRL_WORK = 1, CTRL_EXIT = 2, CTRL_GROUPS = 64 };
constexpr int DEV_BAD_SEQLEN = 1;
constexpr int DEV_TIMEOUT = 2;
// Limit of the end-of-kernel drains (MMAs still running, TMA fills not yet consumed):
// never the caller's shorter limit, so that an aborted CTA frees TMEM and exits only
// after its asynchronous work has completed.
constexpr uint64_t DRAIN_NS = 2000000000ull;

enum : int { MODE_DENSE = 0, MODE_STRATIFIED = 1, MODE_SYSTEMATIC = 2, MODE_IID = 3 };

// Workspace carve-up (byte offsets, each 256-aligned).
struct WsLayout {
    size_t ctrl, qt, w, ctot, cexp, cmax, cpre, dpart_o, dpart_ml, total;
    int n_pad, nch, ns_max;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline WsLayout ws_layout(int B, int H_q, int H_kv, int d, int n_max, bool dense)
{
    WsLayout L{};
    L.n_pad = (int)align_up((size_t)n_max, CHUNK);
    L.nch = L.n_pad / CHUNK;
    L.ns_max = (n_max + DENSE_UNIT - 1) / DENSE_UNIT;  // dense partials per sequence
    const size_t BH = (size_t)B * H_q;
    size_t off = 0;
    L.ctrl = off;
    off = align_up(off + sizeof(int) * (CTRL_GROUPS + (size_t)B * H_kv), 256);
    L.qt = off;  // Bernoulli qK^T: the ternary query draws, bf16 [B*H_q][d]
    off = align_up(off + BH * (size_t)d * sizeof(uint16_t), 256);
    if (!dense) {
        L.w = off;    off = align_up(off + BH * L.n_pad * sizeof(float), 256);
        L.ctot = off; off = align_up(off + BH * L.nch * sizeof(float), 256);
        L.cexp = off; off = align_up(off + BH * L.nch * sizeof(int), 256);
        L.cmax = off; off = align_up(off + BH * L.nch * sizeof(float), 256);
        L.cpre = off; off = align_up(off + BH * L.nch * sizeof(uint64_t), 256);
        L.dpart_o = L.dpart_ml = 0;
    } else {
        L.dpart_o = off;  off = align_up(off + BH * L.ns_max * d * sizeof(float), 256);
        L.dpart_ml = off; off = align_up(off + BH * L.ns_max * 2 * sizeof(float), 256);
        L.w = L.ctot = L.cexp = L.cmax = L.cpre = 0;
    }
    L.total = off;
    return L;
}

struct Params {
    const uint16_t *q, *k, *v;   // bf16 bits
    const int32_t *seq_lens;
    float *out;
    int32_t *idx_out;
    int32_t *ctrl;
    float *w;         // [B*H_q][n_pad] fp32 weights 2^(s log2e - c_t), c_t the chunk's scale
    float *ctot;      // [B*H_q][nch] chunk totals of w (chunk scale)
    int32_t *cexp;    // [B*H_q][nch] c_t = ceil of the chunk's maximum of s log2e
    float *cmax;      // [B*H_q][nch] the chunk's maximum of s log2e (fast fp32 scores)
    uint64_t *cpre;   // [B*H_q][nch] value stage: fixed-point CDF prefix (very long sequences)
    float *dpart_o, *dpart_ml;
    int B, H_q, H_kv, n_max, n_pad, nch, ns_max;
    int L;            // keys per work unit (sampled path) or split length (dense), multiple of 64
    int S, mode;
    int xdedup;       // value stage: the group's heads share V loads (thread-block clusters)
    int nstages;      // single-pass cluster kernel: stages of its ring
    int out_bf16;     // out is bf16 (each fp32 result rounded once), else fp32
    uint64_t seed;
    double rS;        // fp64 value nearest 1/S
    float k2_hi, k2_lo;  // scale*log2(e) as an unevaluated fp32 sum
    float tau2;       // re-scoring window below the maximum (log2 units)
    uint64_t wait_ns; // bounded-wait limit of the main loops (santa_set_wait_limit)
    unsigned long long *tl;  // timeline stamps (a build with SANTA_TIMELINE only; else NULL)
    int tl_rows;             // rows of 16 stamps that tl holds
};

// Timeline of a call, for reading where the time goes: a build with -DSANTA_TIMELINE
// (libsanta_timeline.so, see timeline.py) writes %globaltimer stamps into Params::tl,
// 16 per row: score kernel and cluster kernel CTAs in rows [0, 1024), value-stage CTAs in
// rows 1024 + (b * H_q + h).  The normal build compiles the stamps out.
#ifdef SANTA_TIMELINE
#define SANTA_STAMP(row, col)                                                                        \
    do {                                                                                             \
        if (p.tl && (int)(row) < p.tl_rows) p.tl[(size_t)(row) * 16 + (col)] = globaltimer_ns();     \
    } while (0)
#else
#define SANTA_STAMP(row, col) ((void)0)
#endif
constexpr int TL_VALUE_ROW0 = 1024;

// out[i] = v, as fp32 or rounded once to bf16 (round to nearest, ties to even).
__device__ __forceinline__ void store_out(const Params &p, size_t i, float v)
{
    if (p.out_bf16)
        reinterpret_cast<__nv_bfloat16 *>(p.out)[i] = __float2bfloat16_rn(v);
    else
        p.out[i] = v;
}

// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the barrier phase with the given parity; give up after limit_ns.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Global stores with an L2 cache policy (data the next kernel reads back).
__device__ __forceinline__ void st_hint(float *a, float v, uint64_t pol)
{
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(a), "f"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_hint(int *a, int v, uint64_t pol)
{
    asm volatile("st.global.L2::cache_hint.s32 [%0], %1, %2;" ::"l"(a), "r"(v), "l"(pol) : "memory");
}

// Drop the 128-byte L2 lines lying wholly inside [base, base + bytes) without writing
// them back: their data becomes undefined.  For scratch that has been read for the last
// time, so that dirty lines are not evicted to DRAM later.  Threads tid of nt share it.
__device__ __forceinline__ void l2_discard_range(const void *base, size_t bytes, int tid, int nt)
{
    const size_t g = __cvta_generic_to_global(base);
    const size_t a0 = (g + 127) & ~(size_t)127;
    const size_t a1 = (g + bytes) & ~(size_t)127;
    for (size_t a = a0 + (size_t)tid * 128; a < a1; a += (size_t)nt * 128)
        asm volatile("discard.global.L2 [%0], 128;" ::"l"(a) : "memory");
}

// Fetch the 128-byte line holding p into L2 (no register result, nothing waits on it).
__device__ __forceinline__ void prefetch_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(__cvta_generic_to_global(p)));
}

// ------------------------------------------------------------------ arithmetic

// bf16 halves of a 32-bit word -> fp32, exact.
__device__ __forceinline__ float bf16lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Error-free transformations (Knuth's TwoSum, Dekker's Fast2Sum, FMA-based TwoProd):
// s + e == a + b exactly.  The _rn intrinsics keep the compiler from contracting or
// reassociating them.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e)
{
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

__device__ __forceinline__ void fast_two_sum(float a, float b, float &s, float &e)
{
    s = __fadd_rn(a, b);
    e = __fsub_rn(b, __fsub_rn(s, a));
}

// Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
// 1, 2, 3", SC'11): 10 rounds of two 64x64->128 multiplies, key bumped by the Weyl
// constants between rounds.
__device__ __forceinline__ void philox4x64_10(uint64_t c[4], uint64_t k0, uint64_t k1)
{
    const uint64_t M0 = 0xD2E7470EE14C6C93ULL, M1 = 0xCA5A826395121157ULL;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += 0x9E3779B97F4A7C15ULL;
            k1 += 0xBB67AE8584CAA73BULL;
        }
        const uint64_t hi0 = __umul64hi(M0, c[0]), lo0 = M0 * c[0];
        const uint64_t hi1 = __umul64hi(M1, c[2]), lo1 = M1 * c[2];
        const uint64_t y0 = hi1 ^ c[1] ^ k0, y2 = hi0 ^ c[3] ^ k1;
        c[0] = y0;
        c[1] = lo1;
        c[2] = y2;
        c[3] = lo0;
    }
}

// Top 32 bits of a Philox word, as an exact fp64 uniform in [0, 1).
__device__ __forceinline__ double word_uniform(uint64_t x)
{
    return __dmul_rn(__uint2double_rn((uint32_t)(x >> 32)), 0x1p-32);
}

// floor(t 2^64) of the sample point t = (s + u) rS, u = (word >> 32) 2^-32 the word's
// 32-bit uniform and rS = rs_bits as a positive normal double, bit for bit as IEEE double
// arithmetic evaluates it (u + s, then one multiply rounded to nearest even, then the
// exact scaling by 2^64 truncated) -- but in integers, with no fp64 unit.  For 0 <= s <
// 2^20: (s + u) 2^32 is an exact integer y of at most 52 bits, rS = M 2^(E - 1075) with a
// 53-bit M, and their product P = y M (at most 105 bits) is rounded to 53 bits.
__host__ __device__ inline uint64_t point_fraction(int s, uint64_t word, uint64_t rs_bits)
{
    const uint64_t y = ((uint64_t)(uint32_t)s << 32) | (word >> 32);
    if (y == 0) return 0;
    const uint64_t M = (rs_bits & ((1ull << 52) - 1)) | (1ull << 52);
    const int E = (int)((rs_bits >> 52) & 0x7ff);
#ifdef __CUDA_ARCH__
    const uint64_t hi = __umul64hi(y, M), lo = y * M;
    const int nb = hi ? 128 - __clzll((long long)hi) : 64 - __clzll((long long)lo);
#else
    const unsigned __int128 P = (unsigned __int128)y * M;
    const uint64_t hi = (uint64_t)(P >> 64), lo = (uint64_t)P;
    const int nb = hi ? 128 - __builtin_clzll(hi) : 64 - __builtin_clzll(lo);
#endif
    int r = nb > 53 ? nb - 53 : 0;  // bits rounded off (at most 52)
    uint64_t q = lo;
    if (r > 0) {
        q = (lo >> r) | (hi << (64 - r));
        const uint64_t half = (lo >> (r - 1)) & 1u;                         // the first bit off
        const bool sticky = (lo & ((1ull << (r - 1)) - 1u)) != 0;           // any bit below it
        if (half && (sticky || (q & 1u))) ++q;
        if (q >> 53) {  // rounded up to 2^53
            q >>= 1;
            ++r;
        }
    }
    // t = q 2^(r - 32 + E - 1075), so t 2^64 = q 2^(r + E - 1043) (below 2^64: t < 1)
    const int sh = r + E - 1043;
    return sh >= 0 ? (q << sh) : (sh <= -64 ? 0 : (q >> -sh));
}

// Philox block (blk, b, h, domain) keyed by (seed, 0).
__device__ __forceinline__ void philox_block(uint64_t seed, uint64_t blk, int b, int h, uint64_t dom,
                                             uint64_t out[4])
{
    out[0] = blk;
    out[1] = (uint64_t)b;
    out[2] = (uint64_t)h;
    out[3] = dom;
    philox4x64_10(out, seed, 0);
}

// Sample point t_s of (b, h) for the systematic and stratified modes:
//   systematic  t_s = (u + s) * rS, u from word 0 of block (0, b, h, 2)
//   stratified  t_s = (s + u_s) * rS, u_s from word s%4 of block (s/4, b, h, 1)
// with rS the fp64 value nearest 1/S; u + s is exact, the multiply rounds once.
__device__ __forceinline__ double sample_point(int mode, uint64_t seed, int b, int h, int s, double rS)
{
    uint64_t rnd[4];
    if (mode == MODE_SYSTEMATIC) {
        philox_block(seed, 0, b, h, 2, rnd);
        return __dmul_rn(__dadd_rn(word_uniform(rnd[0]), (double)s), rS);
    }
    philox_block(seed, (uint64_t)(s / 4), b, h, 1, rnd);
    return __dmul_rn(__dadd_rn((double)s, word_uniform(rnd[s % 4])), rS);
}

// ------------------------------------------------------------------ CDF fixed point
//
// The CDF pieces are unsigned 64-bit fixed-point numbers with FIX_F fraction bits in a
// power-of-two scale: a chunk total t (fp32, scale 2^-c_t) enters its split (scale
// 2^-c_r, c_r >= c_t) as round(t * 2^(FIX_F + c_t - c_r)).  Sums of these integers are
// exact and order-independent, so patches by integer atomics stay deterministic, and
// no fp64 arithmetic (slow on this part) is needed anywhere on the path.  Chunk totals
// are at most 32 (weights <= 1), split totals at most 512 * 2^40 = 2^49, and a
// sequence's total in the global scale at most 2^19 * 2^40 = 2^59.
constexpr int FIX_F = 40;

// round(x * 2^e) for a non-negative fp32 x (NaN and Inf are treated as 0).  The
// result must stay below 2^64: here x * 2^e <= 2^49 always.
__device__ __forceinline__ uint64_t fixp(float x, int e)
{
    const uint32_t u = __float_as_uint(x);
    const int ex = (int)((u >> 23) & 0xffu);
    if (ex == 0 || ex == 0xff || (u >> 31)) return 0;  // zero, subnormal, Inf/NaN, negative
    const uint64_t m = (u & 0x7fffffu) | 0x800000u;     // x = m * 2^(ex - 150)
    const int sh = ex - 150 + e;
    if (sh >= 0) return sh < 40 ? (m << sh) : 0;       // (cannot happen for totals <= 2^9)
    if (sh < -25) return 0;
    return (m + (1ull << (-sh - 1))) >> (-sh);
}

// d << k, saturating at 2^64 - 1 (0 <= k).
__device__ __forceinline__ uint64_t shl_sat(uint64_t d, int k)
{
    if (k == 0) return d;
    if (k >= 64) return d ? ~0ull : 0ull;
    return (d >> (64 - k)) ? ~0ull : (d << k);
}

// round(d / 2^k) (0 <= k); 0 for k >= 64.
__device__ __forceinline__ uint64_t shr_round(uint64_t d, int k)
{
    if (k == 0) return d;
    if (k >= 64) return 0;
    return (d >> k) + ((d >> (k - 1)) & 1ull);
}

// 2^e as an fp32 for any integer e (0 below the normal range, +Inf above it).
__device__ __forceinline__ float exp2i(int e)
{
    if (e < -126) return 0.f;
    if (e > 127) return __int_as_float(0x7f800000);
    return __int_as_float((e + 127) << 23);
}

// fp32 -> int32 key with the same order (negative values: all bits but the sign flipped),
// for integer reductions and atomics on floats; and its inverse.
__device__ __forceinline__ int fkey(float x)
{
    const int i = __float_as_int(x);
    return i >= 0 ? i : (i ^ 0x7fffffff);
}
__device__ __forceinline__ float fkey_inv(int k) { return __int_as_float(k >= 0 ? k : (k ^ 0x7fffffff)); }

__device__ __forceinline__ void set_dev_error(int32_t *ctrl, int bits)
{
    atomicOr(ctrl + CTRL_ERR, bits);
}

}  // namespace santa
