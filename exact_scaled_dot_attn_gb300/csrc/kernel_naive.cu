// Naive three-pass attention forward: the textbook pipeline with the N x N score and
// probability matrices materialised in device memory, as the comparison baseline of the fused
// kernels ("Naive Attention Kernel", sections "1. Standard Attention: Step by Step", "2. HBM
// Traffic Analysis" and "3. Naive CUDA Implementation"; "Tensor Parallelism with CUDA -
// Standard Attention", section "The Naive HBM Algorithm"):
//
//   pass 1  naive_qk_kernel       reads Q, K   writes S = sm_scale * Q K^T          fp32
//   pass 2  naive_softmax_kernel  reads S      writes P = softmax(S + mask), lse    fp16, fp32
//   pass 3  naive_pv_kernel       reads P, V   writes O = P V                       fp16
//
// Every score of every head is computed, stored and read back, including those the causal
// mask or the key lengths exclude (the naive algorithm materialises the whole matrix); the
// mask is applied in the softmax pass, which also writes the zeros of the excluded entries.
// S is kept in fp32 (the naive page's kernel sketch works on fp32 scores) because fp16 scores
// of peaked rows would lose the parity tolerance; P is fp16 ("FP16 storage, FP32
// accumulation" of the standard-attention page). The scale is folded into pass 1 (the
// standard-attention page's qkKernel) and the mask into the softmax pass (the naive page's
// fused scale/mask/softmax kernel), so S is written once and read once, P written once and
// read once.
//
// The two products are tiled over shared memory and run on the warp-level tensor core
// instruction (mma.sync m16n8k16, fp16 in, fp32 accumulate): the point of this baseline is the
// traffic of the materialised matrices, not slow arithmetic, so its time is set by memory.
// Rows of S and P are padded to a multiple of 128 columns (Np), so every tile is aligned and
// the padded columns of P hold zeros.
#include "attn_internal.h"

#include <math.h>

#include "warp_mma_ops.cuh"

namespace attn {
namespace {

using namespace warpmma;

constexpr int kTile = 128;     // rows (and, in pass 1, keys) per CTA tile
constexpr int kThreads = 256;  // 8 warps x 16 rows
constexpr int kKeyChunk = 64;  // keys per step of pass 3
constexpr int kSmThreads = 256; // softmax pass: 8 warps, one row each

__host__ __device__ inline long long padded_cols(int N) { return (static_cast<long long>(N) + kTile - 1) / kTile * kTile; }

// Rows [r0, r0 + rows) of a [n, D] fp16 matrix into a swizzled shared tile with cp.async;
// rows >= n are zero-filled.
template <int D>
__device__ __forceinline__ void load_rows(__half *s, const __half *g, int r0, int rows, int n)
{
    constexpr int CPR = D / 8; // 16-byte chunks per row
    for (int c = threadIdx.x; c < rows * CPR; c += kThreads) {
        const int r = c / CPR, ch = c % CPR;
        const int gr = r0 + r;
        const bool ok = gr < n;
        cp_async16(s + swz<D>(r, ch), g + static_cast<size_t>(ok ? gr : 0) * D + ch * 8, ok);
    }
}

// Pass 1: the 128 x 128 tile (row tile rt, key tile ct) of S = sm_scale * Q K^T of one head.
template <int D>
__global__ void __launch_bounds__(kThreads)
    naive_qk_kernel(const __half *__restrict__ q, const __half *__restrict__ k, float *__restrict__ s,
                    int N, long long Np, int n_tiles, float sm_scale)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __half *sQ = reinterpret_cast<__half *>(smem_raw); // [128][D]
    __half *sK = sQ + kTile * D;                        // [128][D]
    const long long blk = blockIdx.x;
    const int ct = static_cast<int>(blk % n_tiles);
    const int rt = static_cast<int>((blk / n_tiles) % n_tiles);
    const long long bh = blk / (static_cast<long long>(n_tiles) * n_tiles);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    load_rows<D>(sQ, q + bh * N * D, rt * kTile, kTile, N);
    load_rows<D>(sK, k + bh * N * D, ct * kTile, kTile, N);
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();

    const int wrow0 = warp * 16;
    float acc[kTile / 8][4];
#pragma unroll
    for (int nb = 0; nb < kTile / 8; ++nb)
        acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.f;
#pragma unroll
    for (int kb = 0; kb < D / 16; ++kb) {
        unsigned a[4];
        ldsm_x4(a[0], a[1], a[2], a[3], sQ + swz<D>(wrow0 + (lane & 15), kb * 2 + (lane >> 4)));
#pragma unroll
        for (int np = 0; np < kTile / 16; ++np) {
            unsigned b0, b1, b2, b3;
            const int r = np * 16 + (lane & 7) + ((lane >> 4) << 3);
            ldsm_x4(b0, b1, b2, b3, sK + swz<D>(r, kb * 2 + ((lane >> 3) & 1)));
            mma16816(acc[2 * np], a, b0, b1);
            mma16816(acc[2 * np + 1], a, b2, b3);
        }
    }
    // thread: rows wrow0 + lane / 4 (+ 8), columns 2 (lane % 4) + {0, 1} of every 8-column block
    const int ra = rt * kTile + wrow0 + (lane >> 2);
    float *srow_a = s + (bh * N + ra) * Np + ct * kTile + ((lane & 3) << 1);
    float *srow_b = srow_a + 8 * Np;
#pragma unroll
    for (int nb = 0; nb < kTile / 8; ++nb) {
        if (ra < N)
            *reinterpret_cast<float2 *>(srow_a + nb * 8) = make_float2(acc[nb][0] * sm_scale, acc[nb][1] * sm_scale);
        if (ra + 8 < N)
            *reinterpret_cast<float2 *>(srow_b + nb * 8) = make_float2(acc[nb][2] * sm_scale, acc[nb][3] * sm_scale);
    }
}

// (m, l) of two parts of a row merged: the softmax normaliser against the larger maximum.
__device__ __forceinline__ void merge_ml(float &m, float &l, float m2, float l2)
{
    const float mn = fmaxf(m, m2);
    if (mn == -INFINITY)
        return; // both parts empty
    l = l * expf(m - mn) + l2 * expf(m2 - mn);
    m = mn;
}

// Pass 2: one warp per row of S (eight rows per CTA). The allowed keys of row i of batch b
// are j < lim = min(L_b, i + 1 under the causal mask); the row's maximum and normaliser come
// from one online pass over them (the naive page's fused softmax: running maximum, normaliser
// rescaled when the maximum grows), then P = exp(s - m) / l is written over the whole padded
// row (zeros outside the allowed keys) and lse = m + ln l.
__global__ void __launch_bounds__(kSmThreads)
    naive_softmax_kernel(const float *__restrict__ s, __half *__restrict__ p, float *__restrict__ lse,
                         const int32_t *__restrict__ key_lengths, int H, int N, long long Np, int causal,
                         long long rows)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = static_cast<long long>(blockIdx.x) * (kSmThreads / 32) + warp;
    if (row >= rows)
        return;
    const long long bh = row / N;
    const int i = static_cast<int>(row - bh * N);
    const int b = static_cast<int>(bh / H);
    int lim = N;
    if (key_lengths) {
        const int L = key_lengths[b];
        lim = L < 0 ? 0 : (L > N ? N : L);
    }
    if (causal)
        lim = min(lim, i + 1);
    const float *srow = s + row * Np;
    __half *prow = p + row * Np;

    // online maximum and normaliser of this lane's allowed entries, 4 consecutive per step
    float m = -INFINITY, l = 0.f;
    for (int j = lane * 4; j < lim; j += 128) {
        const float4 x4 = *reinterpret_cast<const float4 *>(srow + j);
        float xs[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
            xs[e] = j + e < lim ? xs[e] : -INFINITY;
        const float bm = fmaxf(fmaxf(xs[0], xs[1]), fmaxf(xs[2], xs[3])); // xs[0] is allowed
        if (bm > m) {
            l *= expf(m - bm);
            m = bm;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e)
            l += expf(xs[e] - m);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
        const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
        merge_ml(m, l, m2, l2);
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;

    for (long long j = lane * 4; j < Np; j += 128) {
        float pv[4] = {0.f, 0.f, 0.f, 0.f};
        if (j < lim) {
            const float4 x4 = *reinterpret_cast<const float4 *>(srow + j);
            const float xs[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                pv[e] = j + e < lim ? expf(xs[e] - m) * inv : 0.f;
        }
        const __half2 h0 = __floats2half2_rn(pv[0], pv[1]);
        const __half2 h1 = __floats2half2_rn(pv[2], pv[3]);
        uint2 w2;
        w2.x = *reinterpret_cast<const unsigned *>(&h0);
        w2.y = *reinterpret_cast<const unsigned *>(&h1);
        *reinterpret_cast<uint2 *>(prow + j) = w2;
    }
    if (lse && lane == 0)
        lse[row] = l > 0.f ? m + logf(l) : -INFINITY;
}

// Pass 3: rows [rt * 128, rt * 128 + 128) of O = P V for one head, over every (padded) key
// column of P in chunks of 64 keys, double-buffered with cp.async.
template <int D>
__global__ void __launch_bounds__(kThreads)
    naive_pv_kernel(const __half *__restrict__ p, const __half *__restrict__ v, __half *__restrict__ o,
                    int N, long long Np, int n_tiles)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __half *sP = reinterpret_cast<__half *>(smem_raw); // [2][128][64]
    __half *sV = sP + 2 * kTile * kKeyChunk;            // [2][64][D]
    const long long blk = blockIdx.x;
    const int rt = static_cast<int>(blk % n_tiles);
    const long long bh = blk / n_tiles;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const __half *gP = p + (bh * N + static_cast<long long>(rt) * kTile) * Np;
    const __half *gV = v + bh * N * D;
    const int rows = min(kTile, N - rt * kTile);
    const int n_chunks = static_cast<int>(Np / kKeyChunk);

    // P rows of this tile, keys [c0, c0 + 64); rows past N are zero-filled
    auto load_p = [&](__half *dst, int c0) {
        constexpr int CPR = kKeyChunk / 8;
        for (int c = threadIdx.x; c < kTile * CPR; c += kThreads) {
            const int r = c / CPR, ch = c % CPR;
            const bool ok = r < rows;
            cp_async16(dst + swz<kKeyChunk>(r, ch), gP + static_cast<long long>(ok ? r : 0) * Np + c0 + ch * 8, ok);
        }
    };
    load_p(sP, 0);
    load_rows<D>(sV, gV, 0, kKeyChunk, N);
    cp_async_commit();

    const int wrow0 = warp * 16;
    float acc[D / 8][4];
#pragma unroll
    for (int db = 0; db < D / 8; ++db)
        acc[db][0] = acc[db][1] = acc[db][2] = acc[db][3] = 0.f;
    for (int c = 0; c < n_chunks; ++c) {
        const int st = c & 1;
        if (c + 1 < n_chunks) {
            load_p(sP + (st ^ 1) * kTile * kKeyChunk, (c + 1) * kKeyChunk);
            load_rows<D>(sV + (st ^ 1) * kKeyChunk * D, gV, (c + 1) * kKeyChunk, kKeyChunk, N);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const __half *ps = sP + st * kTile * kKeyChunk;
        const __half *vs = sV + st * kKeyChunk * D;
#pragma unroll
        for (int kb = 0; kb < kKeyChunk / 16; ++kb) {
            unsigned a[4];
            ldsm_x4(a[0], a[1], a[2], a[3], ps + swz<kKeyChunk>(wrow0 + (lane & 15), kb * 2 + (lane >> 4)));
#pragma unroll
            for (int dp = 0; dp < D / 16; ++dp) {
                unsigned b0, b1, b2, b3;
                const int r = kb * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                ldsm_x4_t(b0, b1, b2, b3, vs + swz<D>(r, dp * 2 + (lane >> 4)));
                mma16816(acc[2 * dp], a, b0, b1);
                mma16816(acc[2 * dp + 1], a, b2, b3);
            }
        }
        __syncthreads();
    }
    const int ra = rt * kTile + wrow0 + (lane >> 2);
    __half *orow_a = o + (bh * N + ra) * D + ((lane & 3) << 1);
    __half *orow_b = orow_a + 8 * D;
#pragma unroll
    for (int db = 0; db < D / 8; ++db) {
        if (ra < N)
            *reinterpret_cast<__half2 *>(orow_a + db * 8) = __floats2half2_rn(acc[db][0], acc[db][1]);
        if (ra + 8 < N)
            *reinterpret_cast<__half2 *>(orow_b + db * 8) = __floats2half2_rn(acc[db][2], acc[db][3]);
    }
}

template <int D>
cudaError_t launch_naive_d(const FwdParams &prm, float *s, __half *p, cudaStream_t stream)
{
    const long long BH = static_cast<long long>(prm.B) * prm.H;
    const int N = prm.N;
    const long long Np = padded_cols(N);
    const int n_tiles = static_cast<int>(Np / kTile);
    const long long qk_blocks = BH * n_tiles * n_tiles;
    const long long pv_blocks = BH * n_tiles;
    const long long rows = BH * N;
    if (qk_blocks > 0x7fffffffLL || rows > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    const int qk_smem = 2 * kTile * D * static_cast<int>(sizeof(__half));
    const int pv_smem = 2 * (kTile * kKeyChunk + kKeyChunk * D) * static_cast<int>(sizeof(__half));
    cudaError_t err = cudaFuncSetAttribute(naive_qk_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, qk_smem);
    if (err == cudaSuccess)
        err = cudaFuncSetAttribute(naive_pv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, pv_smem);
    if (err != cudaSuccess)
        return err;
    naive_qk_kernel<D><<<static_cast<unsigned>(qk_blocks), kThreads, qk_smem, stream>>>(
        prm.q, prm.k, s, N, Np, n_tiles, prm.sm_scale);
    const long long sm_blocks = (rows + kSmThreads / 32 - 1) / (kSmThreads / 32);
    naive_softmax_kernel<<<static_cast<unsigned>(sm_blocks), kSmThreads, 0, stream>>>(
        s, p, prm.lse, prm.key_lengths, prm.H, N, Np, prm.causal, rows);
    naive_pv_kernel<D><<<static_cast<unsigned>(pv_blocks), kThreads, pv_smem, stream>>>(
        p, prm.v, prm.o, N, Np, n_tiles);
    return cudaGetLastError();
}

} // namespace

long long naive_padded_cols(int N) { return padded_cols(N); }

cudaError_t launch_naive(const FwdParams &p, float *s, __half *pm, cudaStream_t stream)
{
    switch (p.d) {
    case 32: return launch_naive_d<32>(p, s, pm, stream);
    case 64: return launch_naive_d<64>(p, s, pm, stream);
    case 128: return launch_naive_d<128>(p, s, pm, stream);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace attn
