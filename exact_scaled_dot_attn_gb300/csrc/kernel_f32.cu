// Attention forward for fp32 inputs at fp32 accuracy (head dimension 32): the precision of the
// "cuda-reranker" README's fp32 kernel, on the tensor cores it names as its next step.
//
// A tensor-core product of fp32 operands reads 10 fraction bits of each (TF32). Splitting every
// operand x into hi = x rounded to 10 fraction bits and lo = x - hi (exact in fp32, of which the
// tensor core reads the 10 leading fraction bits in turn), a product of two values is formed
// from three TF32 products,
//     a b ~ a_hi b_lo + a_lo b_hi + a_hi b_hi,
// the published error-corrected TF32 method (Ootomo and Yokota, 2022): the term left out,
// a_lo b_lo, and the bits of the lo parts the tensor core does not read stay within 5 * 2^-22
// of |a b|, so the products carry about fp32's precision, and they accumulate in fp32. Both
// products of the attention use it: S = Q K^T and O += P V, with P split the same way.
//
// The tiled recurrence is that of "Self-Attention Kernel & Inference Engine from Scratch"
// ("Online Softmax Formulation"): one CTA owns 64 query rows of one (batch, head); 64-key K/V
// tiles stream through a two-stage cp.async ring; the running row max and normaliser are fp32;
// P stays fp32 (split into TF32 parts for the product, never rounded to 16 bits); O is fp32.
// The split and the products run on the warp-level instruction mma.sync m16n8k8 (tf32), with
// the hi/lo parts formed in registers, so no extra copy of any tile is kept in memory.
// The causal block skip and the all-padding tile skip reduce to stopping the tile loop at the
// last tile with an allowed key. Cross-attention and grouped-query attention: the K/V rows come
// from the query head's key/value head and the causal diagonal moves by Nk - N.
#include "attn_internal.h"

#include <math.h>

#include "warp_mma_ops.cuh"

namespace attn {
namespace {

using namespace warpmma;

constexpr int kD = 32;           // head dimension
constexpr int kBM = 64;          // query rows per CTA: 4 warps x 16 rows
constexpr int kBN = 64;          // keys per K/V tile
constexpr int kThreads = 128;
// floats per shared row, so that the fragment loads of a warp hit distinct banks: 64-bit loads
// of Q and K (a half-warp reads 4 rows x 4 pairs), 32-bit loads of V (4 rows x 8 columns)
constexpr int kStride = kD + 8;  // Q and K
constexpr int kStrideV = kD + 4; // V
constexpr float kLn2f = 0.6931471805599453f;

// x = hi + lo: hi is x rounded to 10 fraction bits (nearest, ties away from zero: half a unit
// of the 10th bit added to the bit pattern, the 13 low bits cleared), so |x - hi| <= 2^-11 |x|;
// lo = x - hi is exact in fp32 and is passed whole (the tensor core reads its sign, exponent
// and 10 leading fraction bits). Finite inputs below 2^127 in magnitude.
__device__ __forceinline__ void split(float x, uint32_t &hi, uint32_t &lo)
{
    hi = (__float_as_uint(x) + 0x1000u) & 0xffffe000u;
    lo = __float_as_uint(x - __uint_as_float(hi));
}

// D[16x8] += A[16x8] * B[8x8], TF32 operands, fp32 accumulators. (Not volatile: it has no
// effect beyond its outputs, so the compiler may interleave products into different
// accumulators; the callers already place independent accumulators between dependent
// products, since one product takes 8 issue cycles of the SMSP and its result is needed by the
// next product into the same accumulator.)
__device__ __forceinline__ void mma_tf32(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, "
        "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Rows [r0, r0 + 64) of a [n, 32] fp32 matrix into a shared tile of row stride STRIDE;
// rows >= n are zero-filled.
template <int STRIDE>
__device__ __forceinline__ void load_tile(float *s, const float *g, int r0, int n)
{
    constexpr int CPR = kD / 4; // 16-byte chunks per row
    for (int c = threadIdx.x; c < kBN * CPR; c += kThreads) {
        const int r = c / CPR, ch = c % CPR;
        const int gr = r0 + r;
        const bool ok = gr < n;
        cp_async16(s + r * STRIDE + ch * 4, g + static_cast<size_t>(ok ? gr : 0) * kD + ch * 4, ok);
    }
}

// Fragment layouts of mma.m16n8k8 (tf32), lane = 4 g + t4:
//   A (16 x 8): a0 (g, t4), a1 (g + 8, t4), a2 (g, t4 + 4), a3 (g + 8, t4 + 4)
//   B (8 x 8):  b0 (k = t4, n = g), b1 (k = t4 + 4, n = g)
//   C (16 x 8): c0, c1 (g, 2 t4 + {0, 1}), c2, c3 (g + 8, 2 t4 + {0, 1})
// Both products take their k index in the order 0, 2, 4, 6, 1, 3, 5, 7 of the underlying
// dimension (k = t4 is element 2 t4, k = t4 + 4 is element 2 t4 + 1), the same for A and B, so
// the sums are unchanged: for S = Q K^T a thread's two Q (or K) elements are adjacent in a row
// and load as one 64-bit access; for O += P V the S accumulator of an 8-key block is the A
// fragment as it stands (a = {c0, c2, c1, c3}) and V is read at rows 2 t4 and 2 t4 + 1.
__global__ void __launch_bounds__(kThreads)
    attn_fwd_f32_kernel(const FwdParams p, int n_qtiles)
{
    extern __shared__ __align__(128) float smem_f[];
    float *sQ = smem_f;                 // [64][kStride]
    float *sK = sQ + kBM * kStride;     // [2][64][kStride]
    float *sV = sK + 2 * kBN * kStride; // [2][64][kStrideV]
    const float *gq = reinterpret_cast<const float *>(p.q);
    const float *gk = reinterpret_cast<const float *>(p.k);
    const float *gv = reinterpret_cast<const float *>(p.v);
    float *go = reinterpret_cast<float *>(p.o);

    const int BH = p.B * p.H;
    // The heaviest query tiles (last under a causal mask) are issued first.
    const int qt = n_qtiles - 1 - static_cast<int>(blockIdx.x / BH);
    const int bh = static_cast<int>(blockIdx.x % BH);
    const int b = bh / p.H;
    const int N = p.N, Nk = p.Nk;
    const int diag = Nk - N; // causal: query i sees keys j <= i + diag
    const int q0 = qt * kBM;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;

    int L = Nk;
    if (p.key_lengths) {
        L = p.key_lengths[b];
        L = L < 0 ? 0 : (L > Nk ? Nk : L);
    }
    int kv_end = L;
    if (p.causal && !p.qrows) // (packed query groups: every tile sees all keys up to L)
        kv_end = max(0, min(kv_end, q0 + kBM + diag));
    const int qdiag = p.qrows ? Nk - p.qrows : diag;
    const int n_tiles = (kv_end + kBN - 1) / kBN;

    const size_t head_off = static_cast<size_t>(bh) * N * kD;
    const int kvh = b * p.Hkv + (bh - b * p.H) / (p.H / p.Hkv);
    const size_t kv_off = static_cast<size_t>(kvh) * Nk * kD;

    load_tile<kStride>(sQ, gq + head_off, q0, N);
    if (n_tiles > 0) {
        load_tile<kStride>(sK, gk + kv_off, 0, Nk);
        load_tile<kStrideV>(sV, gv + kv_off, 0, Nk);
    }
    cp_async_commit();

    const int wrow0 = warp * 16;
    const int row_a = q0 + wrow0 + g; // this thread's rows: row_a and row_a + 8
    const int row_b = row_a + 8;
    const int lim_a = (p.qrows ? row_a % p.qrows : row_a) + qdiag; // causal: last allowed key
    const int lim_b = (p.qrows ? row_b % p.qrows : row_b) + qdiag;
    float o[kD / 8][4];
#pragma unroll
    for (int nb = 0; nb < kD / 8; ++nb)
        o[nb][0] = o[nb][1] = o[nb][2] = o[nb][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY}; // running max of the scaled scores (log2 units)
    float l[2] = {0.f, 0.f};             // this thread's share of the normaliser
    uint32_t qh[kD / 8][4], ql[kD / 8][4];
    const float scale = p.scale_log2;

    for (int t = 0; t < n_tiles; ++t) {
        const int st = t & 1;
        if (t + 1 < n_tiles) {
            load_tile<kStride>(sK + (st ^ 1) * kBN * kStride, gk + kv_off, (t + 1) * kBN, Nk);
            load_tile<kStrideV>(sV + (st ^ 1) * kBN * kStrideV, gv + kv_off, (t + 1) * kBN, Nk);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        if (t == 0) {
#pragma unroll
            for (int kb = 0; kb < kD / 8; ++kb) {
                const float2 qa = *reinterpret_cast<const float2 *>(sQ + (wrow0 + g) * kStride + kb * 8 + 2 * t4);
                const float2 qb = *reinterpret_cast<const float2 *>(sQ + (wrow0 + g + 8) * kStride + kb * 8 + 2 * t4);
                split(qa.x, qh[kb][0], ql[kb][0]);
                split(qb.x, qh[kb][1], ql[kb][1]);
                split(qa.y, qh[kb][2], ql[kb][2]);
                split(qb.y, qh[kb][3], ql[kb][3]);
            }
        }
        const float *ks = sK + st * kBN * kStride;
        const float *vs = sV + st * kBN * kStrideV;
        // S = Q K^T for the 16 x 64 block of this warp: for each 8-wide slice of d, the three
        // products (small terms first) each over the eight 8-key blocks, so that eight
        // independent accumulators lie between two products into the same one
        float s[kBN / 8][4];
#pragma unroll
        for (int nb = 0; nb < kBN / 8; ++nb)
            s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.f;
#pragma unroll
        for (int kb = 0; kb < kD / 8; ++kb) {
            uint32_t bh[kBN / 8][2], bl[kBN / 8][2];
#pragma unroll
            for (int nb = 0; nb < kBN / 8; ++nb) {
                const float2 kr = *reinterpret_cast<const float2 *>(ks + (nb * 8 + g) * kStride + kb * 8 + 2 * t4);
                split(kr.x, bh[nb][0], bl[nb][0]);
                split(kr.y, bh[nb][1], bl[nb][1]);
            }
#pragma unroll
            for (int nb = 0; nb < kBN / 8; ++nb)
                mma_tf32(s[nb], ql[kb], bh[nb][0], bh[nb][1]);
#pragma unroll
            for (int nb = 0; nb < kBN / 8; ++nb)
                mma_tf32(s[nb], qh[kb], bl[nb][0], bl[nb][1]);
#pragma unroll
            for (int nb = 0; nb < kBN / 8; ++nb)
                mma_tf32(s[nb], qh[kb], bh[nb][0], bh[nb][1]);
        }
        // scale into log2 units, mask, running max
        const int kv0 = t * kBN;
        const bool need_mask = (kv0 + kBN > L) ||
                               (p.causal && kv0 + kBN - 1 > (p.qrows ? qdiag : q0 + wrow0 + diag));
        float mx[2] = {m[0], m[1]};
#pragma unroll
        for (int nb = 0; nb < kBN / 8; ++nb) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float x = s[nb][e] * scale;
                if (need_mask) {
                    const int key = kv0 + nb * 8 + 2 * t4 + (e & 1);
                    const int lim = e < 2 ? lim_a : lim_b;
                    if (key >= L || (p.causal && key > lim))
                        x = -INFINITY;
                }
                s[nb][e] = x;
                mx[e >> 1] = fmaxf(mx[e >> 1], x);
            }
        }
        float m_use[2], alpha[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
            // a row without an allowed key so far keeps m = -inf and exponentiates against 0,
            // so masked scores give exactly 0
            m_use[r] = mx[r] == -INFINITY ? 0.f : mx[r];
            alpha[r] = ex2(m[r] - m_use[r]);
            m[r] = mx[r];
            l[r] *= alpha[r];
        }
#pragma unroll
        for (int nb = 0; nb < kD / 8; ++nb) {
            o[nb][0] *= alpha[0];
            o[nb][1] *= alpha[0];
            o[nb][2] *= alpha[1];
            o[nb][3] *= alpha[1];
        }
        // P = 2^(x - m) in fp32, and O += P V with P and V split: per 8-key block the three
        // products each over the four 8-wide slices of d (four independent accumulators
        // between two products into the same one)
#pragma unroll
        for (int kb = 0; kb < kBN / 8; ++kb) {
            const float p0 = ex2(s[kb][0] - m_use[0]), p1 = ex2(s[kb][1] - m_use[0]);
            const float p2 = ex2(s[kb][2] - m_use[1]), p3 = ex2(s[kb][3] - m_use[1]);
            l[0] += p0 + p1;
            l[1] += p2 + p3;
            uint32_t ph[4], pl[4];
            split(p0, ph[0], pl[0]); // (g, key 2 t4)
            split(p2, ph[1], pl[1]); // (g + 8, key 2 t4)
            split(p1, ph[2], pl[2]); // (g, key 2 t4 + 1)
            split(p3, ph[3], pl[3]); // (g + 8, key 2 t4 + 1)
            uint32_t bh[kD / 8][2], bl[kD / 8][2];
#pragma unroll
            for (int nb = 0; nb < kD / 8; ++nb) {
                const float *vr = vs + (kb * 8 + 2 * t4) * kStrideV + nb * 8 + g;
                split(vr[0], bh[nb][0], bl[nb][0]);        // V[key 2 t4][n]
                split(vr[kStrideV], bh[nb][1], bl[nb][1]); // V[key 2 t4 + 1][n]
            }
#pragma unroll
            for (int nb = 0; nb < kD / 8; ++nb)
                mma_tf32(o[nb], pl, bh[nb][0], bh[nb][1]);
#pragma unroll
            for (int nb = 0; nb < kD / 8; ++nb)
                mma_tf32(o[nb], ph, bl[nb][0], bl[nb][1]);
#pragma unroll
            for (int nb = 0; nb < kD / 8; ++nb)
                mma_tf32(o[nb], ph, bh[nb][0], bh[nb][1]);
        }
        __syncthreads();
    }
    cp_async_wait<0>();

    // Epilogue: O / l in fp32, lse (natural log).
    float inv[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
        l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
        inv[r] = l[r] > 0.f ? 1.f / l[r] : 0.f;
    }
#pragma unroll
    for (int nb = 0; nb < kD / 8; ++nb) {
        const int col = nb * 8 + 2 * t4;
        if (row_a < N)
            *reinterpret_cast<float2 *>(go + head_off + static_cast<size_t>(row_a) * kD + col) =
                make_float2(o[nb][0] * inv[0], o[nb][1] * inv[0]);
        if (row_b < N)
            *reinterpret_cast<float2 *>(go + head_off + static_cast<size_t>(row_b) * kD + col) =
                make_float2(o[nb][2] * inv[1], o[nb][3] * inv[1]);
    }
    if (p.lse && t4 == 0) {
        float *lse_head = p.lse + static_cast<size_t>(bh) * N;
        if (row_a < N)
            lse_head[row_a] = l[0] > 0.f ? (m[0] + log2f(l[0])) * kLn2f : -INFINITY;
        if (row_b < N)
            lse_head[row_b] = l[1] > 0.f ? (m[1] + log2f(l[1])) * kLn2f : -INFINITY;
    }
}

} // namespace

cudaError_t launch_f32(const FwdParams &p, cudaStream_t stream)
{
    if (p.d != kD || p.Hkv < 1 || p.H % p.Hkv != 0)
        return cudaErrorInvalidValue;
    const size_t smem = static_cast<size_t>(kBM * kStride + 2 * kBN * kStride + 2 * kBN * kStrideV) * sizeof(float);
    cudaError_t err = cudaFuncSetAttribute(attn_fwd_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess)
        return err;
    const int n_qtiles = (p.N + kBM - 1) / kBM;
    const long long blocks = static_cast<long long>(n_qtiles) * p.B * p.H;
    if (blocks > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    attn_fwd_f32_kernel<<<static_cast<unsigned>(blocks), kThreads, smem, stream>>>(p, n_qtiles);
    return cudaGetLastError();
}

} // namespace attn
