// Decoding kernel: a few query rows (one new token per head, or the packed query heads of a
// grouped-query group) over a long key/value sequence. The attention is the one of the other
// kernels ("Tensor Parallelism with CUDA - Standard Attention", steps 1 to 3, with the running
// maximum and normaliser of "Self-Attention Kernel & Inference Engine from Scratch", "Online
// Softmax Formulation"); only the decomposition differs.
//
// With at most 16 query rows per head there is almost nothing to contract: the work is reading
// K and V once, so the kernel is built for HBM, not for the tensor cores. Each head is handled
// by a thread-block cluster of C CTAs (C = 1, 2, 4 or 8, chosen so the grid fills the SMs). CTA
// c of the cluster streams its contiguous share of the head's 32-key tiles through shared
// memory with cp.async (three stages, 16-byte copies, the tail zero-filled), and keeps the
// running state of every row:
//   scores    lane = key, warp = quarter of the head dimension; the four partial dot products
//             of a key meet in shared memory (fp32; Q is held pre-scaled by sm_scale * log2 e)
//   softmax   warp w takes rows w, w + 4, ...; lane = key: the tile maximum and sum by warp
//             shuffles, P = 2^(s - m), the rescale factor 2^(m_old - m_new) of the row
//   P V       warp w takes 8 of the tile's keys, lane = D / 32 columns, all rows; the four
//             warps' partial outputs are added once at the end
// The CTAs of a cluster then merge their partial (m, l, O) through distributed shared memory
// (the two-block merge of the same section, applied to C blocks), each CTA writing its share of
// the head's output elements. No workspace, no second launch, no waits other than the cluster
// and CTA barriers.
#include "attn_internal.h"

#include <math.h>
#include <mutex>
#include <type_traits>

#include "warp_mma_ops.cuh"

namespace attn {
namespace {

using warpmma::cp_async16;
using warpmma::cp_async_commit;
using warpmma::cp_async_wait;
using warpmma::ex2;

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kKT = 32;        // keys per tile
constexpr int kStages = 3;     // tiles in shared memory (two in flight while one is used)
constexpr int kMaxCluster = 8; // portable cluster size
constexpr float kLn2 = 0.6931471805599453f;

// Shared-memory layout of one CTA (byte offsets). K rows are padded by 16 bytes so the 32
// lanes of a warp reading 32 different rows at the same columns hit distinct banks; V rows are
// read along the row and need no padding.
template <int D, int R> struct DecSmem {
    static constexpr int kKs = D + 8; // K row stride (elements)
    static constexpr int kVs = D;     // V row stride (elements)
    static constexpr int kStageElems = kKT * (kKs + kVs);
    static constexpr int kKv = 0;
    static constexpr int kKvBytes = kStages * kStageElems * 2;
    static constexpr int kQ = kKvBytes;                        // fp32 [R][D]
    static constexpr int kSp = kQ + R * D * 4;                 // fp32 [kWarps][R][kKT]
    static constexpr int kPt = kSp + kWarps * R * kKT * 4;     // fp32 [kKT][R]
    static constexpr int kM = kPt + kKT * R * 4;               // fp32 [R]
    static constexpr int kL = kM + R * 4;                      // fp32 [R]
    static constexpr int kAl = kL + R * 4;                     // fp32 [R]
    static constexpr int kLim = kAl + R * 4;                   // int [R]
    static constexpr int kBytes = kLim + R * 4;
    // after the loop the K/V stages hold the warps' partial outputs, fp32 [kWarps][R][D]
    static_assert(kWarps * R * D * 4 <= kKvBytes, "partial outputs must fit the K/V stages");
    static_assert(kQ % 16 == 0 && kSp % 16 == 0 && kPt % 16 == 0, "16-byte aligned regions");
};

struct DecArgs {
    const void *q, *k, *v;
    void *o;
    float *lse;
    const int32_t *key_lengths;
    int H, Hkv, N, Nk, qrows, causal;
    float scale_log2;
};

template <typename T> struct Elt;
template <> struct Elt<__half> {
    static __device__ __forceinline__ float2 pair(uint32_t w)
    {
        return __half22float2(*reinterpret_cast<const __half2 *>(&w));
    }
    static __device__ __forceinline__ float one(__half x) { return __half2float(x); }
    static __device__ __forceinline__ __half from(float x) { return __float2half_rn(x); }
};
template <> struct Elt<__nv_bfloat16> {
    // a bf16 value is the high half of the fp32 value with the same bits
    static __device__ __forceinline__ float2 pair(uint32_t w)
    {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
    static __device__ __forceinline__ float one(__nv_bfloat16 x) { return __bfloat162float(x); }
    static __device__ __forceinline__ __nv_bfloat16 from(float x) { return __float2bfloat16_rn(x); }
};

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;\n" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;\n" : "=r"(r));
    return r;
}
// Every thread of every CTA of the cluster arrives; shared-memory writes before it are visible
// to the whole cluster after it.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// fp32 at shared-memory address `addr` (of this CTA's layout) in CTA `rank` of the cluster.
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr, uint32_t rank)
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(remote) : "r"(addr), "r"(rank));
    float x;
    asm volatile("ld.shared::cluster.f32 %0, [%1];\n" : "=f"(x) : "r"(remote) : "memory");
    return x;
}

__device__ __forceinline__ float warp_max(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// DPL consecutive elements of a shared-memory row as fp32.
template <typename T, int DPL> __device__ __forceinline__ void load_cols(float *f, const T *p)
{
    if constexpr (DPL == 4) {
        const uint2 w = *reinterpret_cast<const uint2 *>(p);
        const float2 a = Elt<T>::pair(w.x), b = Elt<T>::pair(w.y);
        f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    } else if constexpr (DPL == 2) {
        const float2 a = Elt<T>::pair(*reinterpret_cast<const uint32_t *>(p));
        f[0] = a.x; f[1] = a.y;
    } else {
        f[0] = Elt<T>::one(*p);
    }
}

// One head (batch * query head) per cluster; see the file comment. D: head dimension, R: query
// rows per head rounded up to 4, 8 or 16 (rows >= N are padding and are not written).
template <int D, int R, typename T>
__global__ void __launch_bounds__(kThreads, R <= 4 ? 4 : 3) attn_fwd_decode_kernel(DecArgs a)
{
    using L = DecSmem<D, R>;
    constexpr int DQ = D / kWarps; // head-dimension columns per warp in the score phase
    constexpr int DPL = D / 32;    // columns per lane in the P V phase
    constexpr int KPW = kKT / kWarps; // keys per warp in the P V phase
    extern __shared__ __align__(16) unsigned char smem[];
    T *kv = reinterpret_cast<T *>(smem + L::kKv);
    float *qs = reinterpret_cast<float *>(smem + L::kQ);
    float *sp = reinterpret_cast<float *>(smem + L::kSp);
    float *pt = reinterpret_cast<float *>(smem + L::kPt);
    float *m_s = reinterpret_cast<float *>(smem + L::kM);
    float *l_s = reinterpret_cast<float *>(smem + L::kL);
    float *al_s = reinterpret_cast<float *>(smem + L::kAl);
    int *lim_s = reinterpret_cast<int *>(smem + L::kLim);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = cluster_ctarank();
    const uint32_t C = cluster_nctarank();
    const long long bh = cluster_id_x();
    const int b = static_cast<int>(bh / a.H), h = static_cast<int>(bh % a.H);
    const long long bkv = static_cast<long long>(b) * a.Hkv + h / (a.H / a.Hkv);
    const T *qg = static_cast<const T *>(a.q) + bh * a.N * D;
    const T *kg = static_cast<const T *>(a.k) + bkv * a.Nk * D;
    const T *vg = static_cast<const T *>(a.v) + bkv * a.Nk * D;

    // keys of batch b: j < clamp(key_lengths[b], 0, Nk); under the causal mask row r (query
    // r % qrows of a packed group, else query r) also needs j <= query + Nk - (query rows)
    int klen = a.Nk;
    if (a.key_lengths)
        klen = min(max(a.key_lengths[b], 0), a.Nk);
    if (tid < R) {
        int lim = 0;
        if (tid < a.N) {
            lim = klen;
            if (a.causal) {
                const int nq = a.qrows ? a.qrows : a.N;
                const int qi = a.qrows ? tid % a.qrows : tid;
                const long long c = static_cast<long long>(qi) + a.Nk - nq + 1;
                lim = static_cast<int>(min(static_cast<long long>(lim), max(c, 0LL)));
            }
        }
        lim_s[tid] = lim;
        m_s[tid] = -INFINITY;
        l_s[tid] = 0.f;
    }
    for (int e = tid; e < R * D; e += kThreads) {
        const int r = e / D;
        qs[e] = r < a.N ? Elt<T>::one(qg[e]) * a.scale_log2 : 0.f;
    }
    __syncthreads();
    int n_keys = 0;
#pragma unroll
    for (int r = 0; r < R; ++r)
        n_keys = max(n_keys, lim_s[r]);
    const int n_tiles = (n_keys + kKT - 1) / kKT;
    const int t0 = static_cast<int>(static_cast<long long>(n_tiles) * rank / C);
    const int nt = static_cast<int>(static_cast<long long>(n_tiles) * (rank + 1) / C) - t0;

    // tile t of this CTA (keys (t0 + t) * kKT ...) into stage s; keys >= n_keys read as zero
    auto load_tile = [&](int t, int s) {
        constexpr int CPR = D / 8; // 16-byte chunks per row
        T *ks = kv + s * L::kStageElems;
        T *vs = ks + kKT * L::kKs;
        const int key0 = (t0 + t) * kKT;
        for (int c = tid; c < kKT * CPR; c += kThreads) {
            const int r = c / CPR, ch = c % CPR;
            const int key = key0 + r;
            const bool ok = key < n_keys;
            const long long src = static_cast<long long>(ok ? key : 0) * D + ch * 8;
            cp_async16(ks + r * L::kKs + ch * 8, kg + src, ok);
            cp_async16(vs + r * L::kVs + ch * 8, vg + src, ok);
        }
    };

#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        if (s < nt)
            load_tile(s, s);
        cp_async_commit();
    }

    float acc[R][DPL];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int c = 0; c < DPL; ++c)
            acc[r][c] = 0.f;

    for (int t = 0; t < nt; ++t) {
        cp_async_wait<kStages - 2>(); // this thread's copies of tile t have landed
        __syncthreads();              // everyone's have; tile t - 1 is no longer read
        {
            const int tn = t + kStages - 1;
            if (tn < nt)
                load_tile(tn, tn % kStages);
            cp_async_commit();
        }
        const T *ks = kv + (t % kStages) * L::kStageElems;
        const T *vs = ks + kKT * L::kKs;
        const int key0 = (t0 + t) * kKT;

        // scores: this lane's key, this warp's quarter of the head dimension, every row
        {
            float kf[DQ];
            const T *krow = ks + lane * L::kKs + warp * DQ;
#pragma unroll
            for (int c = 0; c < DQ / 8; ++c) {
                const uint4 w = *reinterpret_cast<const uint4 *>(krow + c * 8);
                const float2 f0 = Elt<T>::pair(w.x), f1 = Elt<T>::pair(w.y);
                const float2 f2 = Elt<T>::pair(w.z), f3 = Elt<T>::pair(w.w);
                kf[c * 8 + 0] = f0.x; kf[c * 8 + 1] = f0.y; kf[c * 8 + 2] = f1.x; kf[c * 8 + 3] = f1.y;
                kf[c * 8 + 4] = f2.x; kf[c * 8 + 5] = f2.y; kf[c * 8 + 6] = f3.x; kf[c * 8 + 7] = f3.y;
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float *qr = qs + r * D + warp * DQ;
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int c = 0; c < DQ; c += 4) {
                    const float4 q4 = *reinterpret_cast<const float4 *>(qr + c);
                    s0 = fmaf(q4.x, kf[c], s0);
                    s1 = fmaf(q4.y, kf[c + 1], s1);
                    s0 = fmaf(q4.z, kf[c + 2], s0);
                    s1 = fmaf(q4.w, kf[c + 3], s1);
                }
                sp[(warp * R + r) * kKT + lane] = s0 + s1;
            }
        }
        __syncthreads();

        // softmax step of rows warp, warp + 4, ...: lane = key
#pragma unroll
        for (int r = warp; r < R; r += kWarps) {
            float s = sp[(0 * R + r) * kKT + lane] + sp[(1 * R + r) * kKT + lane] +
                      sp[(2 * R + r) * kKT + lane] + sp[(3 * R + r) * kKT + lane];
            if (key0 + lane >= lim_s[r])
                s = -INFINITY;
            const float m_old = m_s[r];
            const float l_old = l_s[r];
            const float m_new = fmaxf(m_old, warp_max(s));
            const float m_use = m_new == -INFINITY ? 0.f : m_new; // no key yet: P = 0
            const float p = ex2(s - m_use);
            const float sum = warp_sum(p);
            pt[lane * R + r] = p;
            __syncwarp();
            if (lane == 0) {
                const float alpha = ex2(m_old - m_use);
                al_s[r] = alpha;
                m_s[r] = m_new;
                l_s[r] = l_old * alpha + sum;
            }
        }
        __syncthreads();

        // O = alpha * O + P V over this warp's keys; lane = columns lane * DPL ...
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float al = al_s[r];
#pragma unroll
            for (int c = 0; c < DPL; ++c)
                acc[r][c] *= al;
        }
#pragma unroll
        for (int jj = 0; jj < KPW; ++jj) {
            const int j = warp * KPW + jj;
            float vf[DPL];
            load_cols<T, DPL>(vf, vs + j * L::kVs + lane * DPL);
            const float *pj = pt + j * R;
#pragma unroll
            for (int r = 0; r < R; r += 4) {
                const float4 p4 = *reinterpret_cast<const float4 *>(pj + r);
#pragma unroll
                for (int c = 0; c < DPL; ++c) {
                    acc[r][c] = fmaf(p4.x, vf[c], acc[r][c]);
                    acc[r + 1][c] = fmaf(p4.y, vf[c], acc[r + 1][c]);
                    acc[r + 2][c] = fmaf(p4.z, vf[c], acc[r + 2][c]);
                    acc[r + 3][c] = fmaf(p4.w, vf[c], acc[r + 3][c]);
                }
            }
        }
    }
    cp_async_wait<0>();
    __syncthreads(); // every stage read; the stages now hold the warps' partial outputs

    float *ob = reinterpret_cast<float *>(smem + L::kKv); // fp32 [kWarps][R][D]
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int c = 0; c < DPL; ++c)
            ob[(warp * R + r) * D + lane * DPL + c] = acc[r][c];
    __syncthreads();
    for (int e = tid; e < R * D; e += kThreads)
        ob[e] = ob[e] + ob[R * D + e] + ob[2 * R * D + e] + ob[3 * R * D + e];
    __syncwarp();   // the cluster barrier is taken by whole warps
    cluster_sync(); // every CTA's (m, l, O) is complete and visible to the cluster

    // merge of the cluster's partials: this CTA's share of the head's output elements
    const uint32_t m_addr = static_cast<uint32_t>(__cvta_generic_to_shared(m_s));
    const uint32_t l_addr = static_cast<uint32_t>(__cvta_generic_to_shared(l_s));
    const uint32_t o_addr = static_cast<uint32_t>(__cvta_generic_to_shared(ob));
    T *og = static_cast<T *>(a.o) + bh * a.N * D;
    for (int e = static_cast<int>(rank) * kThreads + tid; e < a.N * D; e += kThreads * static_cast<int>(C)) {
        const int r = e / D, col = e % D;
        float M = -INFINITY;
        for (uint32_t i = 0; i < C; ++i)
            M = fmaxf(M, ld_cluster_f32(m_addr + r * 4, i));
        float out = 0.f, lse = -INFINITY;
        if (M != -INFINITY) {
            float Lsum = 0.f, Osum = 0.f;
            for (uint32_t i = 0; i < C; ++i) {
                const float w = ex2(ld_cluster_f32(m_addr + r * 4, i) - M);
                Lsum = fmaf(ld_cluster_f32(l_addr + r * 4, i), w, Lsum);
                Osum = fmaf(ld_cluster_f32(o_addr + e * 4, i), w, Osum);
            }
            out = Osum / Lsum;
            lse = (M + log2f(Lsum)) * kLn2;
        }
        og[e] = Elt<T>::from(out);
        if (col == 0 && a.lse)
            a.lse[bh * a.N + r] = lse;
    }
    __syncwarp();
    cluster_sync(); // no CTA leaves while another still reads its shared memory
}

// Per device and configuration: the dynamic shared memory attribute is set and the largest
// cluster size that the device can place is known (0: not looked up yet).
constexpr int kMaxDevices = 64;
std::mutex g_cfg_mutex;
int g_cfg_cmax[kMaxDevices][3][3][2];
int g_cfg_per_sm[kMaxDevices][3][3][2];

template <int D, int R, typename T>
cudaError_t launch_cfg(const FwdParams &p, cudaStream_t stream)
{
    auto kernel = attn_fwd_decode_kernel<D, R, T>;
    constexpr int smem = DecSmem<D, R>::kBytes;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    const int di = D == 32 ? 0 : D == 64 ? 1 : 2;
    const int ri = R == 4 ? 0 : R == 8 ? 1 : 2;
    const int ti = std::is_same<T, __half>::value ? 0 : 1;
    int cmax, per_sm;
    {
        std::lock_guard<std::mutex> lock(g_cfg_mutex);
        cmax = g_cfg_cmax[dev][di][ri][ti];
        per_sm = g_cfg_per_sm[dev][di][ri][ti];
        if (cmax == 0) {
            err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (err != cudaSuccess)
                return err;
            err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem);
            if (err != cudaSuccess)
                return err;
            if (per_sm < 1)
                return cudaErrorInvalidConfiguration;
            // the largest cluster the device can co-schedule with this footprint
            cmax = kMaxCluster;
            for (; cmax > 1; cmax >>= 1) {
                cudaLaunchConfig_t probe = {};
                probe.gridDim = dim3(static_cast<unsigned>(cmax));
                probe.blockDim = dim3(kThreads);
                probe.dynamicSmemBytes = smem;
                cudaLaunchAttribute at[1];
                at[0].id = cudaLaunchAttributeClusterDimension;
                at[0].val.clusterDim.x = static_cast<unsigned>(cmax);
                at[0].val.clusterDim.y = 1;
                at[0].val.clusterDim.z = 1;
                probe.attrs = at;
                probe.numAttrs = 1;
                int n = 0;
                if (cudaOccupancyMaxActiveClusters(&n, kernel, &probe) == cudaSuccess && n >= 1)
                    break;
                (void)cudaGetLastError(); // a refused size leaves no error behind
            }
            g_cfg_cmax[dev][di][ri][ti] = cmax;
            g_cfg_per_sm[dev][di][ri][ti] = per_sm;
        }
    }
    int sms = 0;
    err = device_sm_count(&sms);
    if (err != cudaSuccess)
        return err;
    // Cluster size: double it while the whole grid still fits in one wave of resident CTAs
    // and every CTA keeps at least four key tiles.
    const long long BH = static_cast<long long>(p.B) * p.H;
    const long long tiles = (static_cast<long long>(p.Nk) + kKT - 1) / kKT;
    int C = 1;
    while (C < cmax && BH * C * 2 <= static_cast<long long>(sms) * per_sm && tiles >= 8LL * C &&
           BH * C * 2 <= 0x7fffffffLL)
        C *= 2;

    DecArgs args;
    args.q = p.q;
    args.k = p.k;
    args.v = p.v;
    args.o = p.o;
    args.lse = p.lse;
    args.key_lengths = p.key_lengths;
    args.H = p.H;
    args.Hkv = p.Hkv;
    args.N = p.N;
    args.Nk = p.Nk;
    args.qrows = p.qrows;
    args.causal = p.causal;
    args.scale_log2 = p.scale_log2;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(BH * C));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = C > 1 ? 1 : 0; // C = 1: every CTA is a cluster of its own
    return cudaLaunchKernelEx(&cfg, kernel, args);
}

template <int D, typename T> cudaError_t launch_rows(const FwdParams &p, cudaStream_t stream)
{
    if (p.N <= 4)
        return launch_cfg<D, 4, T>(p, stream);
    if (p.N <= 8)
        return launch_cfg<D, 8, T>(p, stream);
    return launch_cfg<D, 16, T>(p, stream);
}

template <typename T> cudaError_t launch_dtype(const FwdParams &p, cudaStream_t stream)
{
    switch (p.d) {
    case 32: return launch_rows<32, T>(p, stream);
    case 64: return launch_rows<64, T>(p, stream);
    case 128: return launch_rows<128, T>(p, stream);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace

cudaError_t launch_decode(const FwdParams &p, cudaStream_t stream)
{
    if (p.N < 1 || p.N > kDecodeMaxRows || p.B * static_cast<long long>(p.H) > 0x7fffffffLL)
        return cudaErrorInvalidValue;
    if (p.dtype == kDtypeF16)
        return launch_dtype<__half>(p, stream);
    if (p.dtype == kDtypeBF16)
        return launch_dtype<__nv_bfloat16>(p, stream);
    return cudaErrorInvalidValue;
}

} // namespace attn
