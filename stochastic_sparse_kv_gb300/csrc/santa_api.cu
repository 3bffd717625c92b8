// santa_api.cu -- the C ABI of libsanta.so (declared in include/santa.h): argument
// checks, workspace carve-up, split planning and kernel dispatch.  No allocation, no
// host synchronisation (except santa_device_status), no CPU fallback.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/santa.h"
#include "santa_cluster.cuh"
#include "santa_dense.cuh"
#include "santa_gather.cuh"
#include "santa_kernels.h"
#include "santa_score.cuh"

namespace santa {

int score_smem_bytes(int D, int G, int B)
{
    (void)G;
    return score_smem(D, B).total;
}

int gather_smem_bytes(int D, int G, int S, int nch_used, int mode, bool xdedup, int nth)
{
    return gather_smem(D, G, S, nch_used, mode, xdedup, nth).total;
}

int dense_smem_bytes(int D, int G, int B)
{
    return dense_smem(D, G, B).total;
}

int cluster_smem_bytes(int D, int G, int LW, int S, int mode, int C, int ns)
{
    return cluster_smem(D, G, LW, S, mode, C, ns).total;
}



// ---------------------------------------------------------------- points kernels

__global__ void santa_points_kernel(int B, int H_q, int S, int mode, uint64_t seed, double rS, double *t)
{
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const size_t total = (size_t)B * H_q * S;
    if (i >= total) return;
    const int s = (int)(i % S);
    const int h = (int)((i / S) % H_q);
    const int b = (int)(i / ((size_t)S * H_q));
    t[i] = sample_point(mode, seed, b, h, s, rS);
}

// iid: one CTA per (b, h) sorts its S draws (bitonic, in shared memory).
__global__ void santa_points_iid_kernel(int B, int H_q, int S, uint64_t seed, double *t)
{
    __shared__ unsigned keys[SMAX];
    const int bh = blockIdx.x;
    const int b = bh / H_q, h = bh % H_q;
    int Sp = 1;
    while (Sp < S) Sp <<= 1;
    for (int s = threadIdx.x; s < Sp; s += blockDim.x) {
        unsigned u = 0xffffffffu;
        if (s < S) {
            uint64_t rnd[4];
            philox_block(seed, (uint64_t)(s / 4), b, h, 3, rnd);
            u = (unsigned)(rnd[s % 4] >> 32);
        }
        keys[s] = u;
    }
    __syncthreads();
    for (int k = 2; k <= Sp; k <<= 1)
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int s = threadIdx.x; s < Sp; s += blockDim.x) {
                const int q = s ^ j;
                if (q > s) {
                    const bool asc = (s & k) == 0;
                    const unsigned x = keys[s], y = keys[q];
                    if ((x > y) == asc) {
                        keys[s] = y;
                        keys[q] = x;
                    }
                }
            }
            __syncthreads();
        }
    for (int s = threadIdx.x; s < S; s += blockDim.x)
        t[(size_t)bh * S + s] = __dmul_rn(__uint2double_rn(keys[s]), 0x1p-32);
}

// Bernoulli qK^T ("Stochastic Sparse Attention for Memory-Bound Inference", abstract,
// last sentences: stochastic ternary queries sparsify the score stage).  One warp per
// (b, h): a = max |q_i| over the head, then for each feature i the top 32 bits x of
// Philox word i%4 of block (i/4, b, h, 4) keep sign(q_i) * a when x * 2^-32 < |q_i| / a,
// compared as x * a < |q_i| * 2^32 (both products exact in fp64), else 0.  E[q~] = q.
__global__ void santa_ternary_kernel(int BH, int H_q, int D, uint64_t seed, const uint16_t *q, uint16_t *qt)
{
    const int wid = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5), lane = threadIdx.x & 31;
    if (wid >= BH) return;
    const int b = wid / H_q, h = wid % H_q;
    const uint16_t *qh = q + (size_t)wid * D;
    uint16_t *qo = qt + (size_t)wid * D;
    // the largest magnitude: for non-negative bf16 values the order of the bit patterns is
    // that of the values (NaN patterns, above 0x7f80, are left out)
    uint32_t amax = 0;
    for (int i = lane; i < D; i += 32) {
        const uint32_t m = qh[i] & 0x7fffu;
        if (m <= 0x7f80u) amax = max(amax, m);
    }
    amax = __reduce_max_sync(0xffffffffu, amax);
    const double a = (double)__uint_as_float(amax << 16);
    for (int i4 = lane; i4 < D / 4; i4 += 32) {
        uint64_t rnd[4];
        philox_block(seed, (uint64_t)i4, b, h, 4, rnd);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = 4 * i4 + e;
            const uint32_t bits = qh[i];
            const double qi = (double)__uint_as_float((bits & 0x7fffu) << 16);
            const double x = (double)(uint32_t)(rnd[e] >> 32);
            const bool keep = a > 0.0 && __dmul_rn(x, a) < __dmul_rn(qi, 0x1p32);
            qo[i] = keep ? (uint16_t)((bits & 0x8000u) | amax) : (uint16_t)0;
        }
    }
}

const void *points_kernel() { return (const void *)santa_points_kernel; }
const void *points_iid_kernel() { return (const void *)santa_points_iid_kernel; }

// ---------------------------------------------------------------- per-device caches

constexpr int MAX_DEV_STATIC = 64;
std::mutex g_static_mu;
std::atomic<unsigned long long> g_wait_limit_ns{0};  // 0: the default of 2 s
std::atomic<unsigned long long *> g_timeline{nullptr};  // SANTA_TIMELINE builds: stamp buffer
std::atomic<int> g_timeline_rows{0};

namespace {

constexpr int MAX_DEV = 64;
std::mutex g_mu;
int g_sms[MAX_DEV];
int g_optin[MAX_DEV];

struct FnCache {
    const void *fn;
    int dev, smem_set, occ_smem, occ;
};
FnCache g_fn[256];
int g_nfn = 0;

int device_info(int *dev, int *sms, int *optin)
{
    if (cudaGetDevice(dev) != cudaSuccess) return SANTA_ERR_CUDA;
    if (*dev < 0 || *dev >= MAX_DEV) return SANTA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sms[*dev] == 0) {
        int a = 0, b = 0;
        if (cudaDeviceGetAttribute(&a, cudaDevAttrMultiProcessorCount, *dev) != cudaSuccess) return SANTA_ERR_CUDA;
        if (cudaDeviceGetAttribute(&b, cudaDevAttrMaxSharedMemoryPerBlockOptin, *dev) != cudaSuccess)
            return SANTA_ERR_CUDA;
        g_sms[*dev] = a;
        g_optin[*dev] = b;
    }
    *sms = g_sms[*dev];
    *optin = g_optin[*dev];
    return SANTA_OK;
}

// Raise the kernel's dynamic shared-memory limit if needed; return CTAs per SM.
int prepare_fn(const void *fn, int dev, int smem, int threads, int *occ)
{
    std::lock_guard<std::mutex> lk(g_mu);
    FnCache *c = nullptr;
    for (int i = 0; i < g_nfn; ++i)
        if (g_fn[i].fn == fn && g_fn[i].dev == dev) c = &g_fn[i];
    if (!c) {
        if (g_nfn == 256) return SANTA_ERR_UNSUPPORTED;
        c = &g_fn[g_nfn++];
        c->fn = fn;
        c->dev = dev;
        c->smem_set = 0;
        c->occ_smem = -1;
        c->occ = 0;
    }
    if (smem > 48 * 1024 && smem > c->smem_set) {
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return SANTA_ERR_CUDA;
        c->smem_set = smem;
    }
    if (c->occ_smem != smem) {
        int o = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, fn, threads, smem) != cudaSuccess) return SANTA_ERR_CUDA;
        c->occ = o;
        c->occ_smem = smem;
    }
    *occ = c->occ;
    return *occ > 0 ? SANTA_OK : SANTA_ERR_UNSUPPORTED;
}

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

int check_shape(const santa_shape *sh)
{
    if (!sh) return SANTA_ERR_INVALID_ARG;
    if (sh->B < 1 || sh->H_q < 1 || sh->H_kv < 1 || sh->n_max < 1 || sh->d < 1) return SANTA_ERR_INVALID_ARG;
    if (sh->H_q % sh->H_kv != 0) return SANTA_ERR_INVALID_ARG;
    if (!std::isfinite(sh->scale)) return SANTA_ERR_INVALID_ARG;
    const int G = sh->H_q / sh->H_kv;
    if (G != 1 && G != 2 && G != 4 && G != 8) return SANTA_ERR_UNSUPPORTED;
    if (sh->d != 64 && sh->d != 128) return SANTA_ERR_UNSUPPORTED;
    if (sh->B > BMAX || sh->H_q > 1024) return SANTA_ERR_UNSUPPORTED;
    if (sh->n_max > NMAX_LIMIT) return SANTA_ERR_UNSUPPORTED;
    // the kernels address K and V rows with 32-bit tensor-copy coordinates
    if ((long long)sh->B * sh->H_kv * sh->n_max >= (1ll << 31)) return SANTA_ERR_UNSUPPORTED;
    return SANTA_OK;
}

int check_mode_S(int32_t mode_flags, int32_t S)
{
    if (mode_flags & ~(0xff | SANTA_GROUP_DEDUP | SANTA_OUT_BF16 | SANTA_BERNOULLI_QK | SANTA_TWO_PASS))
        return SANTA_ERR_INVALID_ARG;
    const int mode = mode_flags & 0xff;
    if (mode < SANTA_DENSE || mode > SANTA_IID) return SANTA_ERR_INVALID_ARG;
    if (mode != SANTA_DENSE && (S < 1 || S > SMAX)) return SANTA_ERR_INVALID_ARG;
    return SANTA_OK;
}

// Every host-side check of a decode call except those on the workspace: shape, mode, S,
// the tensor pointers and their alignment, and the control block's size.  Nothing is
// enqueued before these pass (santa_decode and santa_decode_static both call it first).
int check_decode_args(const santa_shape *shape, const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *seq_lens, int32_t S, int32_t mode_flags, const float *out,
                      const int32_t *idx_out)
{
    int rc = check_shape(shape);
    if (rc) return rc;
    if ((rc = check_mode_S(mode_flags, S))) return rc;
    if (!q || !k_cache || !v_cache || !seq_lens || !out) return SANTA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(seq_lens, 4) || (idx_out && !aligned(idx_out, 4)))
        return SANTA_ERR_MISALIGNED;
    const WsLayout wl = ws_layout(shape->B, shape->H_q, shape->H_kv, shape->d, shape->n_max,
                                  (mode_flags & 0xff) == SANTA_DENSE);
    if (wl.ctrl + sizeof(int) * (CTRL_GROUPS + (size_t)shape->B * shape->H_kv) > 65536) return SANTA_ERR_UNSUPPORTED;
    return SANTA_OK;
}

// cuTensorMapEncodeTiled from the driver, found once through the runtime (no link
// against libcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult qr{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// Row-major bf16 matrix [rows][D] as a 2-D tensor map with boxes of 64 columns (128
// bytes, the 128-byte swizzle's width) by box_rows rows.
int make_map_bf16(CUtensorMap *map, const void *base, int D, long long rows, int box_rows)
{
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return SANTA_ERR_CUDA;
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SANTA_OK : SANTA_ERR_CUDA;
}

// The single-pass cluster kernel, when it applies: one cluster of C CTAs per (b, KV head),
// the largest C (at most 16) such that the B * H_kv clusters fit the GPU at once, each CTA
// holding at most CL_LWMAX keys and the points of its group (G * S <= 2048) in shared
// memory.  Otherwise (larger batches, longer caches) the score and value stages run as
// two launches.
struct ClusterPlan {
    int C, LW, ns, smem;
};

struct ClusterOcc {
    const void *fn;
    int dev, C, smem, nclus;
};
ClusterOcc g_cocc[512];
int g_ncocc = 0;

// Clusters of C CTAs (smem bytes each) of kernel fn resident at once on device dev.
int max_active_clusters(const void *fn, int dev, int C, int smem)
{
    {
        std::lock_guard<std::mutex> lk(g_mu);
        for (int i = 0; i < g_ncocc; ++i)
            if (g_cocc[i].fn == fn && g_cocc[i].dev == dev && g_cocc[i].C == C && g_cocc[i].smem == smem)
                return g_cocc[i].nclus;
    }
    int occ = 0;
    if (prepare_fn(fn, dev, smem, CL_NT, &occ)) return 0;
    if (C > 8 && cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)C);
    cfg.blockDim = dim3(CL_NT);
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int nclus = 0;
    if (cudaOccupancyMaxActiveClusters(&nclus, fn, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        nclus = 0;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_ncocc < 512) g_cocc[g_ncocc++] = ClusterOcc{fn, dev, C, smem, nclus};
    return nclus;
}

bool plan_cluster(const santa_shape *shape, int S, int32_t mode_flags, int dev, int sms, int optin, ClusterPlan *pl)
{
    const int mode = mode_flags & 0xff;
    if (mode == SANTA_DENSE || (mode_flags & (SANTA_GROUP_DEDUP | SANTA_TWO_PASS))) return false;
    const int D = shape->d, G = shape->H_q / shape->H_kv;
    const long long groups = (long long)shape->B * shape->H_kv;
    if (G * S > 2048 || groups > sms) return false;
    const void *fn = (D == 128) ? kernel_d128(KIND_CLUSTER, G) : kernel_d64(KIND_CLUSTER, G);
    if (!fn) return false;
    const int units = (shape->n_max + SC_M - 1) / SC_M;
    for (int C = (int)(sms / groups < CL_MAXC ? sms / groups : CL_MAXC); C >= 1; --C) {
        const int LW = (units + C - 1) / C * SC_M;
        if (LW > CL_LWMAX) return false;  // (a smaller C only needs more keys per CTA)
        int ns = cluster_max_stages(D), smem = 0;
        for (; ns >= cluster_min_stages(D); --ns) {
            smem = cluster_smem_bytes(D, G, LW, S, mode, C, ns);
            if (smem <= optin) break;
        }
        if (ns < cluster_min_stages(D)) return false;
        if (max_active_clusters(fn, dev, C, smem) < groups) continue;
        pl->C = C;
        pl->LW = LW;
        pl->ns = ns;
        pl->smem = smem;
        return true;
    }
    return false;
}

}  // namespace
}  // namespace santa

using namespace santa;

extern "C" {

int santa_version(void) { return 10000; }

const char *santa_status_string(int status)
{
    switch (status) {
    case SANTA_OK: return "ok";
    case SANTA_ERR_INVALID_ARG: return "invalid argument";
    case SANTA_ERR_MISALIGNED: return "pointer not aligned (16 bytes for tensors, 256 for the workspace)";
    case SANTA_ERR_WORKSPACE: return "workspace missing or too small";
    case SANTA_ERR_UNSUPPORTED: return "outside the supported limits (d in {64,128}, G in {1,2,4,8}, B <= 1024, "
                                      "n_max <= 524288, S <= 4096, shared memory)";
    case SANTA_ERR_CUDA: return "CUDA runtime error";
    case SANTA_ERR_DEVICE: return "device reported an error (bad seq_lens or a barrier timeout)";
    case SANTA_ERR_SCRATCH: return "the problem needs more scratch than the static buffer of santa_decode_static holds";
    default: return "unknown status";
    }
}

int santa_workspace_size(const santa_shape *shape, int32_t S, int32_t mode, size_t *bytes)
{
    int rc = check_shape(shape);
    if (rc) return rc;
    if ((rc = check_mode_S(mode, S))) return rc;
    if (!bytes) return SANTA_ERR_INVALID_ARG;
    *bytes = ws_layout(shape->B, shape->H_q, shape->H_kv, shape->d, shape->n_max, (mode & 0xff) == SANTA_DENSE).total;
    return SANTA_OK;
}

int santa_workspace_init(void *workspace, size_t workspace_bytes, void *stream)
{
    if (!workspace) return SANTA_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return SANTA_ERR_MISALIGNED;
    const size_t n = workspace_bytes < 256 ? workspace_bytes : 256;
    if (n < sizeof(int) * 4) return SANTA_ERR_WORKSPACE;
    // The control block is CTRL_GROUPS words plus one counter per group; the caller's
    // workspace may be shared across shapes, so clear every counter word it can hold
    // up to the first data region (a conservative 64 KiB bound).
    size_t ctrl = workspace_bytes < (size_t)65536 ? workspace_bytes : (size_t)65536;
    ctrl = ctrl / 4 * 4;
    if (cudaMemsetAsync(workspace, 0, ctrl, (cudaStream_t)stream) != cudaSuccess) return SANTA_ERR_CUDA;
    return SANTA_OK;
}

int santa_decode(const santa_shape *shape, const void *q, const void *k_cache, const void *v_cache,
                 const int32_t *seq_lens, int32_t S, int32_t mode_flags, uint64_t seed, float *out, int32_t *idx_out,
                 void *workspace, size_t workspace_bytes, void *stream)
{
    int rc = check_decode_args(shape, q, k_cache, v_cache, seq_lens, S, mode_flags, out, idx_out);
    if (rc) return rc;
    const int32_t mode = mode_flags & 0xff;
    if (!workspace) return SANTA_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return SANTA_ERR_MISALIGNED;
    const bool dense = (mode == SANTA_DENSE);
    const WsLayout wl = ws_layout(shape->B, shape->H_q, shape->H_kv, shape->d, shape->n_max, dense);
    if (workspace_bytes < wl.total) return SANTA_ERR_WORKSPACE;

    int dev, sms, optin;
    if ((rc = device_info(&dev, &sms, &optin))) return rc;
    const int D = shape->d, G = shape->H_q / shape->H_kv;
    // keys per work unit: SC_M (sampled); DENSE_UNIT times 4, 2 or 1 (dense), the largest
    // that still leaves every SM a dozen splits (fewer partials for the merge to read)
    int L = SC_M;
    if (dense) {
        L = DENSE_UNIT;
        for (int f = 4; f > 1; f /= 2) {
            const int Lf = DENSE_UNIT * f;
            if ((long long)shape->B * shape->H_kv * ((shape->n_max + Lf - 1) / Lf) >= 12LL * sms) {
                L = Lf;
                break;
            }
        }
    }
    Params p{};
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    // Bernoulli qK^T: every step scores with the heads' ternary query draws, which a
    // first launch writes into the workspace (after every check below has passed)
    const bool ternary = (mode_flags & SANTA_BERNOULLI_QK) != 0;
    const void *q_user = q;
    if (ternary) q = ws + wl.qt;
    p.q = static_cast<const uint16_t *>(q);
    p.k = static_cast<const uint16_t *>(k_cache);
    p.v = static_cast<const uint16_t *>(v_cache);
    p.seq_lens = seq_lens;
    p.out = out;
    p.idx_out = dense ? nullptr : idx_out;
    p.ctrl = reinterpret_cast<int32_t *>(ws + wl.ctrl);
    if (!dense) {
        p.w = reinterpret_cast<float *>(ws + wl.w);
        p.ctot = reinterpret_cast<float *>(ws + wl.ctot);
        p.cexp = reinterpret_cast<int32_t *>(ws + wl.cexp);
        p.cmax = reinterpret_cast<float *>(ws + wl.cmax);
        p.cpre = reinterpret_cast<uint64_t *>(ws + wl.cpre);
    } else {
        p.dpart_o = reinterpret_cast<float *>(ws + wl.dpart_o);
        p.dpart_ml = reinterpret_cast<float *>(ws + wl.dpart_ml);
    }
    p.B = shape->B;
    p.H_q = shape->H_q;
    p.H_kv = shape->H_kv;
    p.n_max = shape->n_max;
    p.n_pad = wl.n_pad;
    p.nch = wl.nch;
    p.ns_max = wl.ns_max;
    p.L = L;
    p.S = dense ? 1 : S;
    p.mode = mode;
    p.out_bf16 = (mode_flags & SANTA_OUT_BF16) ? 1 : 0;
    p.seed = seed;
    p.rS = 1.0 / (double)p.S;
    const float scale = shape->scale != 0.f ? shape->scale : (float)(1.0 / std::sqrt((double)D));
    const double k2 = (double)scale * 1.4426950408889634;  // scale * log2(e)
    p.k2_hi = (float)k2;
    p.k2_lo = (float)(k2 - (double)p.k2_hi);
    p.tau2 = (float)(3.0 * 1.4426950408889634);  // re-score keys within e^-3 of the maximum
    const unsigned long long wlim = g_wait_limit_ns.load(std::memory_order_relaxed);
    p.wait_ns = wlim ? wlim : 2000000000ull;
    p.tl = g_timeline.load(std::memory_order_relaxed);
    p.tl_rows = p.tl ? g_timeline_rows.load(std::memory_order_relaxed) : 0;

    ClusterPlan cp{};
    const bool single = plan_cluster(shape, p.S, mode_flags, dev, sms, optin, &cp);
    if (single) {
        // one launch: the single-pass cluster kernel (keys per CTA in Params::L)
        const void *fc = (D == 128) ? kernel_d128(KIND_CLUSTER, G) : kernel_d64(KIND_CLUSTER, G);
        p.L = cp.LW;
        p.nstages = cp.ns;
        const long long krows = (long long)shape->B * shape->H_kv * shape->n_max;
        CUtensorMap tm_k, tm_kt, tm_q;
        if ((rc = make_map_bf16(&tm_k, k_cache, D, krows, SC_M))) return rc;
        if ((rc = make_map_bf16(&tm_kt, k_cache, D, krows, SC_BOX_ROWS))) return rc;
        if ((rc = make_map_bf16(&tm_q, q, D, (long long)shape->B * shape->H_q, G))) return rc;
        if (ternary) {
            const int BH = shape->B * shape->H_q;
            santa_ternary_kernel<<<(unsigned)((BH + 7) / 8), 256, 0, (cudaStream_t)stream>>>(
                BH, shape->H_q, shape->d, seed, static_cast<const uint16_t *>(q_user),
                reinterpret_cast<uint16_t *>(ws + wl.qt));
            if (cudaGetLastError() != cudaSuccess) return SANTA_ERR_CUDA;
        }
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3((unsigned)((long long)shape->B * shape->H_kv * cp.C));
        cfg.blockDim = dim3(CL_NT);
        cfg.dynamicSmemBytes = (size_t)cp.smem;
        cfg.stream = (cudaStream_t)stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)cp.C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        void *cargs[] = {&p, &tm_k, &tm_kt, &tm_q};
        if (cudaLaunchKernelExC(&cfg, fc, cargs) != cudaSuccess) return SANTA_ERR_CUDA;
        return SANTA_OK;
    }
    const int kind = dense ? KIND_DENSE : KIND_SCORE;
    const void *fn = (D == 128) ? kernel_d128(kind, G) : kernel_d64(kind, G);
    if (!fn) return SANTA_ERR_UNSUPPORTED;
    const int smem = dense ? dense_smem_bytes(D, G, shape->B) : score_smem_bytes(D, G, shape->B);
    if (smem > optin) return SANTA_ERR_UNSUPPORTED;
    const int threads = dense ? DN_NT : SC_NT;
    int occ = 0;
    if ((rc = prepare_fn(fn, dev, smem, threads, &occ))) return rc;
    const void *fn2 = nullptr;
    int smem2 = 0, nth2 = NT;
    if (!dense) {
        p.xdedup = ((mode_flags & SANTA_GROUP_DEDUP) && gather_xdedup(G, p.S)) ? 1 : 0;
        // at most one head per SM and long sequences: the wide team (four times the threads
        // on each phase's loops over chunks, and the chunk arrays in shared memory up to
        // 2.5 times as many chunks; measured slower than the narrow team at 1024 chunks,
        // faster at 4096)
        nth2 = NT;
        if (!p.xdedup && (long long)shape->B * shape->H_q <= sms && p.nch > NCH_WIDE_MIN &&
            gather_smem_bytes(D, G, p.S, p.nch, mode, false, NT_WIDE) <= optin)
            nth2 = NT_WIDE;
        const int kind2 = KIND_GATHER + (p.xdedup ? GATHER_XD : 0) + (mode == MODE_IID ? GATHER_IID : 0) +
                          (nth2 == NT_WIDE ? GATHER_WIDE : 0);
        fn2 = (D == 128) ? kernel_d128(kind2, G) : kernel_d64(kind2, G);
        smem2 = gather_smem_bytes(D, G, p.S, p.nch, mode, p.xdedup != 0, nth2);
        if (smem2 > optin) return SANTA_ERR_UNSUPPORTED;
        int occ2 = 0;
        if ((rc = prepare_fn(fn2, dev, smem2, nth2, &occ2))) return rc;
    }
    const long long items = (long long)shape->B * shape->H_kv * ((shape->n_max + L - 1) / L);
    long long grid = (long long)sms * occ;
    if (grid > items) grid = items;
    if (grid < 1) grid = 1;
    void *args[] = {&p};
    const long long krows = (long long)shape->B * shape->H_kv * shape->n_max;
    if (ternary) {
        const int BH = shape->B * shape->H_q;
        santa_ternary_kernel<<<(unsigned)((BH + 7) / 8), 256, 0, (cudaStream_t)stream>>>(
            BH, shape->H_q, shape->d, seed, static_cast<const uint16_t *>(q_user), reinterpret_cast<uint16_t *>(ws + wl.qt));
        if (cudaGetLastError() != cudaSuccess) return SANTA_ERR_CUDA;
    }
    if (dense) {
        // K and V as [B*H_kv*n_max][d] in boxes of a subunit (SC_M rows) and of SC_BOX_ROWS
        // rows (a split's last keys); q in boxes of one group's G heads
        CUtensorMap tm_k, tm_kt, tm_v, tm_vt, tm_q;
        if ((rc = make_map_bf16(&tm_k, k_cache, D, krows, SC_M))) return rc;
        if ((rc = make_map_bf16(&tm_kt, k_cache, D, krows, SC_BOX_ROWS))) return rc;
        if ((rc = make_map_bf16(&tm_v, v_cache, D, krows, SC_M))) return rc;
        if ((rc = make_map_bf16(&tm_vt, v_cache, D, krows, SC_BOX_ROWS))) return rc;
        if ((rc = make_map_bf16(&tm_q, q, D, (long long)shape->B * shape->H_q, G))) return rc;
        void *dargs[] = {&p, &tm_k, &tm_kt, &tm_v, &tm_vt, &tm_q};
        if (cudaLaunchKernel(fn, dim3((unsigned)grid), dim3(DN_NT), dargs, (size_t)smem, (cudaStream_t)stream) !=
            cudaSuccess)
            return SANTA_ERR_CUDA;
        // the merge of the split partials, one CTA per (b, h_q), as a programmatic dependent
        const void *fm = (D == 128) ? kernel_d128(KIND_DMERGE, G) : kernel_d64(KIND_DMERGE, G);
        if (!fm) return SANTA_ERR_UNSUPPORTED;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3((unsigned)(shape->B * shape->H_q));
        cfg.blockDim = dim3((unsigned)(MG_SLICES * D));
        cfg.dynamicSmemBytes = 0;
        cfg.stream = (cudaStream_t)stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelExC(&cfg, fm, args) != cudaSuccess) return SANTA_ERR_CUDA;
    } else {
        // K as [B*H_kv*n_max][d] in boxes of a whole unit (SC_M rows) and of SC_BOX_ROWS rows
        // (a sequence's last unit); q as [B*H_q][d] in boxes of one group's G heads
        CUtensorMap tm_k, tm_kt, tm_q;
        if ((rc = make_map_bf16(&tm_k, k_cache, D, krows, SC_M))) return rc;
        if ((rc = make_map_bf16(&tm_kt, k_cache, D, krows, SC_BOX_ROWS))) return rc;
        if ((rc = make_map_bf16(&tm_q, q, D, (long long)shape->B * shape->H_q, G))) return rc;
        void *sargs[] = {&p, &tm_k, &tm_kt, &tm_q};
        if (cudaLaunchKernel(fn, dim3((unsigned)grid), dim3(SC_NT), sargs, (size_t)smem, (cudaStream_t)stream) !=
            cudaSuccess)
            return SANTA_ERR_CUDA;
    }
    if (!dense) {
        // value stage: one CTA per (b, h_q), a programmatic dependent of the score kernel;
        // the G heads of a group form a cluster when they share V loads
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3((unsigned)(shape->B * shape->H_q));
        cfg.blockDim = dim3((unsigned)nth2);
        cfg.dynamicSmemBytes = (size_t)smem2;
        cfg.stream = (cudaStream_t)stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (p.xdedup) {
            // the group's G heads as one thread-block cluster (they share V loads)
            attr[1].id = cudaLaunchAttributeClusterDimension;
            attr[1].val.clusterDim.x = (unsigned)G;
            attr[1].val.clusterDim.y = 1;
            attr[1].val.clusterDim.z = 1;
            cfg.numAttrs = 2;
        }
        if (cudaLaunchKernelExC(&cfg, fn2, args) != cudaSuccess) return SANTA_ERR_CUDA;
    }
    return SANTA_OK;
}

int santa_call_info(const santa_shape *shape, int32_t S, int32_t mode, int32_t *launches)
{
    int rc = check_shape(shape);
    if (rc) return rc;
    if ((rc = check_mode_S(mode, S))) return rc;
    if (!launches) return SANTA_ERR_INVALID_ARG;
    int dev, sms, optin;
    if ((rc = device_info(&dev, &sms, &optin))) return rc;
    ClusterPlan cp{};
    const bool single = plan_cluster(shape, (mode & 0xff) == SANTA_DENSE ? 1 : S, mode, dev, sms, optin, &cp);
    *launches = (single ? 1 : 2) + ((mode & SANTA_BERNOULLI_QK) ? 1 : 0);
    return SANTA_OK;
}

int santa_timeline_buffer(void *buf, size_t bytes)
{
#ifdef SANTA_TIMELINE
    if (buf && bytes < (size_t)16 * 8 * TL_VALUE_ROW0) return SANTA_ERR_INVALID_ARG;
    if (buf && !aligned(buf, 8)) return SANTA_ERR_MISALIGNED;
    const size_t rows = bytes / (16 * 8);
    g_timeline_rows.store(buf ? (int)std::min<size_t>(rows, 1u << 30) : 0, std::memory_order_relaxed);
    g_timeline.store(static_cast<unsigned long long *>(buf), std::memory_order_relaxed);
    return SANTA_OK;
#else
    (void)buf;
    (void)bytes;
    return SANTA_ERR_UNSUPPORTED;
#endif
}

int santa_set_wait_limit(uint64_t limit_ns)
{
    g_wait_limit_ns.store((unsigned long long)limit_ns, std::memory_order_relaxed);
    return SANTA_OK;
}

int santa_sample_points(int32_t B, int32_t H_q, int32_t S, int32_t mode, uint64_t seed, double *t_out,
                        void *stream)
{
    if (B < 1 || H_q < 1 || S < 1 || S > SMAX || !t_out) return SANTA_ERR_INVALID_ARG;
    if (mode != SANTA_STRATIFIED && mode != SANTA_SYSTEMATIC && mode != SANTA_IID) return SANTA_ERR_INVALID_ARG;
    if (!aligned(t_out, 8)) return SANTA_ERR_MISALIGNED;
    const double rS = 1.0 / (double)S;
    cudaError_t e;
    if (mode == SANTA_IID) {
        void *args[] = {&B, &H_q, &S, &seed, &t_out};
        e = cudaLaunchKernel(points_iid_kernel(), dim3((unsigned)(B * H_q)), dim3(256), args, 0,
                             (cudaStream_t)stream);
    } else {
        const size_t total = (size_t)B * H_q * S;
        void *args[] = {&B, &H_q, &S, &mode, &seed, (void *)&rS, &t_out};
        e = cudaLaunchKernel(points_kernel(), dim3((unsigned)((total + 255) / 256)), dim3(256), args, 0,
                             (cudaStream_t)stream);
    }
    return e == cudaSuccess ? SANTA_OK : SANTA_ERR_CUDA;
}

// The static scratch of santa_decode_static on the current device (defined below), or
// NULL when no static call has run on it yet.
static int static_scratch_ptr(void **ptr, bool create);

int santa_ternary_query(int32_t B, int32_t H_q, int32_t d, const void *q, uint64_t seed, void *q_out,
                        void *stream)
{
    if (B < 1 || H_q < 1 || !q || !q_out) return SANTA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return SANTA_ERR_UNSUPPORTED;
    if ((long long)B * H_q > (1ll << 24)) return SANTA_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(q_out, 16)) return SANTA_ERR_MISALIGNED;
    const int BH = B * H_q;
    santa_ternary_kernel<<<(unsigned)((BH + 7) / 8), 256, 0, (cudaStream_t)stream>>>(
        BH, H_q, d, seed, static_cast<const uint16_t *>(q), static_cast<uint16_t *>(q_out));
    return cudaGetLastError() == cudaSuccess ? SANTA_OK : SANTA_ERR_CUDA;
}

int santa_device_status(void *workspace, int32_t *code, void *stream)
{
    if (!code) return SANTA_ERR_INVALID_ARG;
    if (!workspace) {
        // the static scratch of santa_decode_static on the current device
        const int rc = static_scratch_ptr(&workspace, false);
        if (rc) return rc;
        if (!workspace) {  // no static call has run on this device: nothing to report
            *code = 0;
            return SANTA_OK;
        }
    }
    cudaStream_t s = (cudaStream_t)stream;
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess) return SANTA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SANTA_ERR_CUDA;
    *code = v;
    if (v != 0) {
        if (cudaMemsetAsync(workspace, 0, sizeof v, s) != cudaSuccess) return SANTA_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return SANTA_ERR_CUDA;
        return SANTA_ERR_DEVICE;
    }
    return SANTA_OK;
}


// ---------------------------------------------------------------- santa_decode_static

// The scratch buffer of santa_decode_static: a file-scope device array, so that callers
// that may not allocate device memory can still run a decode step.  Host code must not
// use its name as an address: the device address comes from cudaGetSymbolAddress, once
// per device, with that device current.  Like every __device__ variable without an
// initialiser it starts zeroed, so its error word reads 0 before the first call.
static __device__ __align__(256) unsigned char g_static_scratch[SANTA_STATIC_SCRATCH_BYTES];

namespace {
void *g_static_ptr[santa::MAX_DEV_STATIC];
}

// The device address of the scratch on the current device.  With create, the first
// call on a device looks it up (cudaGetSymbolAddress); without, *ptr is NULL until then.
static int static_scratch_ptr(void **ptr, bool create)
{
    *ptr = nullptr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SANTA_ERR_CUDA;
    if (dev < 0 || dev >= santa::MAX_DEV_STATIC) return SANTA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(santa::g_static_mu);
    if (!g_static_ptr[dev] && create) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return SANTA_ERR_CUDA;
        g_static_ptr[dev] = p;
    }
    *ptr = g_static_ptr[dev];
    return SANTA_OK;
}

int santa_decode_static(const santa_shape *shape, const void *q, const void *k_cache, const void *v_cache,
                        const int32_t *seq_lens, int32_t S, int32_t mode, uint64_t seed, float *out,
                        int32_t *idx_out, void *stream)
{
    // every argument check first: an invalid call enqueues nothing
    size_t need = 0;
    int rc = santa_workspace_size(shape, S, mode, &need);
    if (rc) return rc;
    if (need > SANTA_STATIC_SCRATCH_BYTES) return SANTA_ERR_SCRATCH;
    if ((rc = santa::check_decode_args(shape, q, k_cache, v_cache, seq_lens, S, mode, out, idx_out))) return rc;
    void *ws = nullptr;
    if ((rc = static_scratch_ptr(&ws, true))) return rc;
    // The work counters of the control block start at zero on every call (they may hold
    // anything after a call that gave up early).  Word 0, the device error word, is kept:
    // santa_device_status(NULL, ...) reads and clears it.
    const size_t ctrl = santa::align_up(sizeof(int) * (santa::CTRL_GROUPS + (size_t)shape->B * shape->H_kv), 256);
    if (cudaMemsetAsync(static_cast<uint8_t *>(ws) + sizeof(int), 0, ctrl - sizeof(int), (cudaStream_t)stream) !=
        cudaSuccess)
        return SANTA_ERR_CUDA;
    return santa_decode(shape, q, k_cache, v_cache, seq_lens, S, mode, seed, out, idx_out, ws,
                        SANTA_STATIC_SCRATCH_BYTES, stream);
}

}  // extern "C"
