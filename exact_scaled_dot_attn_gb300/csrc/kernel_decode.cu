// Decoding kernel: a few query rows (one new token per head, or the packed query heads of a
// grouped-query group) over a long key/value sequence. The attention is the one of the other
// kernels ("Tensor Parallelism with CUDA - Standard Attention", steps 1 to 3, with the running
// maximum and normaliser of "Self-Attention Kernel & Inference Engine from Scratch", "Online
// Softmax Formulation"); only the decomposition differs.
//
// With at most 16 query rows per head the work is reading K and V once: the kernel is built to
// keep HBM busy. Each head is handled by a thread-block cluster of C CTAs (C = 1, 2, 4 or 8,
// chosen so the grid fits one wave of resident CTAs). CTA c of the cluster streams its
// contiguous share of the head's 64-key tiles through shared memory with cp.async (three
// stages, 16-byte copies, the rows of a tile XOR-swizzled in 16-byte chunks, keys past the end
// zero-filled). All four warps hold the head's 16 query rows (rows past N are zero) and warp w
// takes keys 16 w .. 16 w + 15 of every tile, with its own running maximum, normaliser and
// output: the two products of a tile are warp-level tensor-core instructions (mma.sync m16n8k16,
// 16-bit inputs, fp32 accumulation; P rounded to the input type), which keeps the instruction
// count per key far below the time its bytes take to arrive. After the last tile the four warps
// are merged in shared memory and the CTAs of the cluster merge their (m, l, O) through
// distributed shared memory (the two-block merge of the same section, applied to 4 C blocks),
// each CTA writing its share of the head's output elements. No workspace, no second launch,
// no waits other than the cluster and CTA barriers.
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
using warpmma::ldsm_x4;
using warpmma::ldsm_x4_t;
using warpmma::swz;

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kRows = 16;      // query rows per head in every warp (the M of the MMA)
constexpr int kKT = 64;        // keys per tile; warp w takes keys 16 w .. 16 w + 15
constexpr int kStages = 3;     // tiles in shared memory (two in flight while one is used)
constexpr int kMaxCluster = 8; // portable cluster size
constexpr float kLn2 = 0.6931471805599453f;

// Shared-memory layout of one CTA (byte offsets). K and V tiles are [kKT][D] and Q is [16][D],
// each row's 16-byte chunks XOR-swizzled by its row index (warpmma::swz) so that the eight
// rows an ldmatrix phase reads fall into different banks.
template <int D> struct DecSmem {
    static constexpr int kTileBytes = kKT * D * 2;      // one K or one V tile
    static constexpr int kStageBytes = 2 * kTileBytes;  // K, then V
    static constexpr int kKv = 0;
    static constexpr int kKvBytes = kStages * kStageBytes;
    static constexpr int kQ = kKvBytes;                  // [16][D]
    static constexpr int kMw = kQ + kRows * D * 2;       // fp32 [kWarps][16] per-warp maxima
    static constexpr int kLw = kMw + kWarps * kRows * 4; // fp32 [kWarps][16] per-warp sums
    static constexpr int kM = kLw + kWarps * kRows * 4;  // fp32 [16] the CTA's maxima
    static constexpr int kL = kM + kRows * 4;            // fp32 [16] the CTA's sums
    static constexpr int kLim = kL + kRows * 4;          // int [16] key limit of every row
    static constexpr int kBytes = kLim + kRows * 4;
    // after the last tile the stages hold the warps' outputs, fp32 [kWarps][16][D], then the
    // CTA's, fp32 [16][D]
    static constexpr int kOw = 0;
    static constexpr int kOb = kWarps * kRows * D * 4;
    static_assert(kOb + kRows * D * 4 <= kKvBytes, "partial outputs must fit the K/V stages");
};

struct DecArgs {
    const void *q, *k, *v;
    void *o;
    float *lse;
    const int32_t *key_lengths;
    int H, Hkv, N, Nk, qrows, causal;
    float scale_log2;
};

// D[16x8] += A[16x16] * B[16x8] with 16-bit inputs of type T and fp32 accumulators, and the
// packing of two fp32 values into one A-fragment register of type T.
template <typename T> struct Mma;
template <> struct Mma<__half> {
    static __device__ __forceinline__ void run(float *c, const unsigned *a, unsigned b0, unsigned b1)
    {
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, "
                     "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
                     : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                     : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    static __device__ __forceinline__ unsigned pack(float lo, float hi)
    {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<unsigned *>(&h);
    }
    static __device__ __forceinline__ __half from(float x) { return __float2half_rn(x); }
};
template <> struct Mma<__nv_bfloat16> {
    static __device__ __forceinline__ void run(float *c, const unsigned *a, unsigned b0, unsigned b1)
    {
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, "
                     "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
                     : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                     : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    static __device__ __forceinline__ unsigned pack(float lo, float hi)
    {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<unsigned *>(&h);
    }
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

// One head (batch * query head) per cluster; see the file comment. D: head dimension.
template <int D, typename T>
__global__ void __launch_bounds__(kThreads, 2) attn_fwd_decode_kernel(DecArgs a)
{
    using L = DecSmem<D>;
    constexpr int CPR = D / 8; // 16-byte chunks per row
    extern __shared__ __align__(1024) unsigned char smem[];
    T *kvs = reinterpret_cast<T *>(smem + L::kKv);
    T *qsm = reinterpret_cast<T *>(smem + L::kQ);
    float *mw = reinterpret_cast<float *>(smem + L::kMw);
    float *lw = reinterpret_cast<float *>(smem + L::kLw);
    float *m_s = reinterpret_cast<float *>(smem + L::kM);
    float *l_s = reinterpret_cast<float *>(smem + L::kL);
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
    if (tid < kRows) {
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
    }
    // the head's query rows (rows >= N read as zero): the oldest copy group
    for (int c = tid; c < kRows * CPR; c += kThreads) {
        const int r = c / CPR, ch = c % CPR;
        const bool ok = r < a.N;
        cp_async16(qsm + swz<D>(r, ch), qg + static_cast<long long>(ok ? r : 0) * D + ch * 8, ok);
    }
    cp_async_commit();
    __syncthreads();
    int n_keys = 0;
#pragma unroll
    for (int r = 0; r < kRows; ++r)
        n_keys = max(n_keys, lim_s[r]);
    const int lim_a = lim_s[lane >> 2], lim_b = lim_s[(lane >> 2) + 8]; // this thread's two rows
    const int n_tiles = (n_keys + kKT - 1) / kKT;
    const int t0 = static_cast<int>(static_cast<long long>(n_tiles) * rank / C);
    const int nt = static_cast<int>(static_cast<long long>(n_tiles) * (rank + 1) / C) - t0;

    // tile t of this CTA (keys (t0 + t) * kKT ...) into stage s; keys >= n_keys read as zero
    auto load_tile = [&](int t, int s) {
        T *ks = kvs + s * (L::kStageBytes / 2);
        T *vs = ks + L::kTileBytes / 2;
        const int key0 = (t0 + t) * kKT;
        for (int c = tid; c < kKT * CPR; c += kThreads) {
            const int r = c / CPR, ch = c % CPR;
            const int key = key0 + r;
            const bool ok = key < n_keys;
            const long long src = static_cast<long long>(ok ? key : 0) * D + ch * 8;
            cp_async16(ks + swz<D>(r, ch), kg + src, ok);
            cp_async16(vs + swz<D>(r, ch), vg + src, ok);
        }
    };

#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
        if (s < nt)
            load_tile(s, s);
        cp_async_commit();
    }
    cp_async_wait<kStages - 1>(); // this thread's Q copies have landed
    __syncthreads();              // everyone's have
    unsigned qf[D / 16][4];
#pragma unroll
    for (int kb = 0; kb < D / 16; ++kb)
        ldsm_x4(qf[kb][0], qf[kb][1], qf[kb][2], qf[kb][3], qsm + swz<D>(lane & 15, kb * 2 + (lane >> 4)));

    // running state of rows lane / 4 and lane / 4 + 8 over this warp's keys (the mma.sync
    // accumulator layout: o[db] holds columns 8 db + 2 (lane % 4) + {0, 1})
    float o[D / 8][4];
#pragma unroll
    for (int db = 0; db < D / 8; ++db)
        o[db][0] = o[db][1] = o[db][2] = o[db][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};

    for (int t = 0; t < nt; ++t) {
        cp_async_wait<kStages - 2>(); // this thread's copies of tile t have landed
        __syncthreads();              // everyone's have; tile t - 1 is no longer read
        {
            const int tn = t + kStages - 1;
            if (tn < nt)
                load_tile(tn, tn % kStages);
            cp_async_commit();
        }
        const T *ks = kvs + (t % kStages) * (L::kStageBytes / 2);
        const T *vs = ks + L::kTileBytes / 2;
        const int key0 = (t0 + t) * kKT + warp * 16;

        // S = Q K^T over this warp's 16 keys
        float s[2][4];
#pragma unroll
        for (int nb = 0; nb < 2; ++nb)
            s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.f;
#pragma unroll
        for (int kb = 0; kb < D / 16; ++kb) {
            unsigned b0, b1, b2, b3;
            const int r = warp * 16 + (lane & 7) + ((lane >> 4) << 3);
            const int ch = kb * 2 + ((lane >> 3) & 1);
            ldsm_x4(b0, b1, b2, b3, ks + swz<D>(r, ch));
            Mma<T>::run(s[0], qf[kb], b0, b1);
            Mma<T>::run(s[1], qf[kb], b2, b3);
        }
        // log2 units, row limits, running maximum
        float mx[2] = {m[0], m[1]};
#pragma unroll
        for (int nb = 0; nb < 2; ++nb) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float x = s[nb][e] * a.scale_log2;
                const int key = key0 + nb * 8 + ((lane & 3) << 1) + (e & 1);
                if (key >= (e < 2 ? lim_a : lim_b))
                    x = -INFINITY;
                s[nb][e] = x;
                mx[e >> 1] = fmaxf(mx[e >> 1], x);
            }
        }
        float m_use[2], alpha[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
            m_use[r] = mx[r] == -INFINITY ? 0.f : mx[r]; // no key yet: P = 0, not NaN
            alpha[r] = ex2(m[r] - m_use[r]);
            m[r] = mx[r];
        }
        // P = 2^(S - m) as the A fragment of the second product; this thread's row sums
        unsigned pf[4];
        float rs[2] = {0.f, 0.f};
#pragma unroll
        for (int nb = 0; nb < 2; ++nb) {
            const float p0 = ex2(s[nb][0] - m_use[0]);
            const float p1 = ex2(s[nb][1] - m_use[0]);
            const float p2 = ex2(s[nb][2] - m_use[1]);
            const float p3 = ex2(s[nb][3] - m_use[1]);
            rs[0] += p0 + p1;
            rs[1] += p2 + p3;
            pf[2 * nb] = Mma<T>::pack(p0, p1);
            pf[2 * nb + 1] = Mma<T>::pack(p2, p3);
        }
#pragma unroll
        for (int r = 0; r < 2; ++r)
            l[r] = l[r] * alpha[r] + rs[r];
        if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
            for (int db = 0; db < D / 8; ++db) {
                o[db][0] *= alpha[0];
                o[db][1] *= alpha[0];
                o[db][2] *= alpha[1];
                o[db][3] *= alpha[1];
            }
        }
        // O += P V over the same 16 keys
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
            unsigned b0, b1, b2, b3;
            const int r = warp * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
            const int ch = dp * 2 + (lane >> 4);
            ldsm_x4_t(b0, b1, b2, b3, vs + swz<D>(r, ch));
            Mma<T>::run(o[2 * dp], pf, b0, b1);
            Mma<T>::run(o[2 * dp + 1], pf, b2, b3);
        }
    }
    cp_async_wait<0>();
    __syncthreads(); // every stage read; the stages now hold the partial outputs

    // this warp's partial (m, l, O) of every row into shared memory
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
        l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
    }
    float *ow = reinterpret_cast<float *>(smem + L::kOw);
    float *ob = reinterpret_cast<float *>(smem + L::kOb);
    const int ra = lane >> 2, rb = ra + 8;
#pragma unroll
    for (int db = 0; db < D / 8; ++db) {
        const int col = db * 8 + ((lane & 3) << 1);
        ow[(warp * kRows + ra) * D + col] = o[db][0];
        ow[(warp * kRows + ra) * D + col + 1] = o[db][1];
        ow[(warp * kRows + rb) * D + col] = o[db][2];
        ow[(warp * kRows + rb) * D + col + 1] = o[db][3];
    }
    if ((lane & 3) == 0) {
        mw[warp * kRows + ra] = m[0];
        mw[warp * kRows + rb] = m[1];
        lw[warp * kRows + ra] = l[0];
        lw[warp * kRows + rb] = l[1];
    }
    __syncthreads();
    // the four warps merged into the CTA's partial
    for (int e = tid; e < kRows * D; e += kThreads) {
        const int r = e / D, col = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w)
            M = fmaxf(M, mw[w * kRows + r]);
        float os = 0.f, ls = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float wt = ex2(mw[w * kRows + r] - M);
                os = fmaf(ow[(w * kRows + r) * D + col], wt, os);
                ls = fmaf(lw[w * kRows + r], wt, ls);
            }
        }
        ob[e] = os;
        if (col == 0) {
            m_s[r] = M;
            l_s[r] = ls;
        }
    }
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
        og[e] = Mma<T>::from(out);
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
int g_cfg_cmax[kMaxDevices][3][2];
int g_cfg_per_sm[kMaxDevices][3][2];

template <int D, typename T>
cudaError_t launch_cfg(const FwdParams &p, cudaStream_t stream)
{
    auto kernel = attn_fwd_decode_kernel<D, T>;
    constexpr int smem = DecSmem<D>::kBytes;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    const int di = D == 32 ? 0 : D == 64 ? 1 : 2;
    const int ti = std::is_same<T, __half>::value ? 0 : 1;
    int cmax, per_sm;
    {
        std::lock_guard<std::mutex> lock(g_cfg_mutex);
        cmax = g_cfg_cmax[dev][di][ti];
        per_sm = g_cfg_per_sm[dev][di][ti];
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
            g_cfg_cmax[dev][di][ti] = cmax;
            g_cfg_per_sm[dev][di][ti] = per_sm;
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

template <typename T> cudaError_t launch_dtype(const FwdParams &p, cudaStream_t stream)
{
    switch (p.d) {
    case 32: return launch_cfg<32, T>(p, stream);
    case 64: return launch_cfg<64, T>(p, stream);
    case 128: return launch_cfg<128, T>(p, stream);
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
