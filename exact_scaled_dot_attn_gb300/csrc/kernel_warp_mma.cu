// Warp-level fused attention forward (mma.sync m16n8k16, fp16 in, fp32 accumulate).
//
// The tiled, fused recurrence of "Self-Attention Kernel & Inference Engine from
// Scratch" (sections "Online Softmax Formulation" and "CUDA Kernel Structure"):
// one CTA owns a tile of 64 query rows of one (batch, head); K and V stream
// through a two-stage shared-memory ring filled by cp.async; S = Q K^T, the
// online-softmax update of the running row max m and normaliser l, the rescale
// of the accumulator and O += P V all happen on chip, so the N x N score matrix
// never reaches memory. The causal block skip of "Engineering Decisions &
// Trade-offs" and the all-padding tile skip of the "cuda-reranker" README both
// reduce to stopping the tile loop at the last tile that holds an allowed key.
//
// This kernel serves every head dimension and length; it is the path for short
// sequences and d = 32, where the work is bound by memory traffic, not by the
// tensor pipe. Long sequences at d in {64, 128} run on the tcgen05 kernel.
#include "attn_internal.h"

#include <math.h>

namespace attn {
namespace {

constexpr int kBM = 64; // query rows per CTA: 4 warps x 16 rows
constexpr int kBN = 64; // keys per K/V tile
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr float kLn2 = 0.6931471805599453f;

// Offset (in halves) of 16-byte chunk `chunk` of row `row` in a [rows][D] tile.
// The chunk index is XOR-ed with bits of the row so that the eight row
// addresses of one ldmatrix phase fall into eight different bank groups.
template <int D> __device__ __forceinline__ int swz(int row, int chunk)
{
    const int x = (D >= 64) ? (row & 7) : ((row >> 1) & 3);
    return row * D + ((chunk ^ x) << 3);
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, bool pred)
{
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    const int n = pred ? 16 : 0; // 0 source bytes: the 16 destination bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N> __device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(unsigned &r0, unsigned &r1, unsigned &r2, unsigned &r3,
                                        const void *p)
{
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(p));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(s));
}
__device__ __forceinline__ void ldsm_x4_t(unsigned &r0, unsigned &r1, unsigned &r2, unsigned &r3,
                                          const void *p)
{
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(p));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(s));
}

// D[16x8] += A[16x16] * B[16x8], fp16 operands, fp32 accumulators.
__device__ __forceinline__ void mma16816(float *c, const unsigned *a, unsigned b0, unsigned b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, "
                 "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 2^x on the special-function unit (ex2.approx; 2^-inf = +0).
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ unsigned pack_half2(float lo, float hi)
{
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<unsigned *>(&h);
}

template <int D>
__global__ void __launch_bounds__(kThreads)
    attn_fwd_warp_mma_kernel(const FwdParams p, int n_qtiles)
{
    constexpr int CPR = D / 8; // 16-byte chunks per row
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __half *sQ = reinterpret_cast<__half *>(smem_raw); // [kBM][D]
    __half *sK = sQ + kBM * D;                           // [2][kBN][D]
    __half *sV = sK + 2 * kBN * D;                       // [2][kBN][D]

    const int BH = p.B * p.H;
    // The heaviest query tiles (last under a causal mask) are issued first.
    const int qt = n_qtiles - 1 - static_cast<int>(blockIdx.x / BH);
    const int bh = static_cast<int>(blockIdx.x % BH);
    const int b = bh / p.H;
    const int N = p.N;
    const int q0 = qt * kBM;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    int L = N;
    if (p.key_lengths) {
        L = p.key_lengths[b];
        L = L < 0 ? 0 : (L > N ? N : L);
    }
    int kv_end = L;
    if (p.causal)
        kv_end = min(kv_end, q0 + kBM);
    const int n_tiles = (kv_end + kBN - 1) / kBN;

    const size_t head_off = static_cast<size_t>(bh) * N * D;
    const __half *gQ = p.q + head_off;
    const __half *gK = p.k + head_off;
    const __half *gV = p.v + head_off;

    // Rows [r0, r0 + kRows) of one head into a swizzled tile; rows >= N are zero-filled.
    auto load_tile = [&](__half *s, const __half *g, int r0, int rows) {
        for (int c = tid; c < rows * CPR; c += kThreads) {
            const int r = c / CPR, ch = c % CPR;
            const int gr = r0 + r;
            const bool ok = gr < N;
            const __half *src = g + static_cast<size_t>(ok ? gr : 0) * D + ch * 8;
            cp_async16(s + swz<D>(r, ch), src, ok);
        }
    };

    load_tile(sQ, gQ, q0, kBM);
    if (n_tiles > 0) {
        load_tile(sK, gK, 0, kBN);
        load_tile(sV, gV, 0, kBN);
    }
    cp_async_commit();

    float o_acc[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i)
        o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
    // Running max (log2 units) and this thread's share of the normaliser, for the
    // two rows the thread holds: lane/4 and lane/4 + 8 of the warp's 16 rows.
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};
    unsigned qf[D / 16][4];

    const int wrow0 = warp * 16;
    const int row_a = q0 + wrow0 + (lane >> 2);
    const int row_b = row_a + 8;

    for (int t = 0; t < n_tiles; ++t) {
        const int st = t & 1;
        if (t + 1 < n_tiles) {
            load_tile(sK + (st ^ 1) * kBN * D, gK, (t + 1) * kBN, kBN);
            load_tile(sV + (st ^ 1) * kBN * D, gV, (t + 1) * kBN, kBN);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        if (t == 0) {
#pragma unroll
            for (int kb = 0; kb < D / 16; ++kb)
                ldsm_x4(qf[kb][0], qf[kb][1], qf[kb][2], qf[kb][3],
                        sQ + swz<D>(wrow0 + (lane & 15), kb * 2 + (lane >> 4)));
        }
        const __half *k_s = sK + st * kBN * D;
        const __half *v_s = sV + st * kBN * D;

        // S = Q K^T for this warp's 16 rows and the tile's 64 keys.
        float s[kBN / 8][4];
#pragma unroll
        for (int nb = 0; nb < kBN / 8; ++nb)
            s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.f;
#pragma unroll
        for (int kb = 0; kb < D / 16; ++kb) {
#pragma unroll
            for (int np = 0; np < kBN / 16; ++np) {
                unsigned b0, b1, b2, b3;
                const int r = np * 16 + (lane & 7) + ((lane >> 4) << 3);
                const int ch = kb * 2 + ((lane >> 3) & 1);
                ldsm_x4(b0, b1, b2, b3, k_s + swz<D>(r, ch));
                mma16816(s[2 * np], qf[kb], b0, b1);
                mma16816(s[2 * np + 1], qf[kb], b2, b3);
            }
        }

        // Scale into log2 units, mask, and update the running max.
        const int kv0 = t * kBN;
        const bool need_mask = (kv0 + kBN > L) || (p.causal && kv0 + kBN - 1 > q0 + wrow0);
        float mx[2] = {m_run[0], m_run[1]};
#pragma unroll
        for (int nb = 0; nb < kBN / 8; ++nb) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float x = s[nb][e] * p.scale_log2;
                if (need_mask) {
                    const int key = kv0 + nb * 8 + ((lane & 3) << 1) + (e & 1);
                    const int row = (e < 2) ? row_a : row_b;
                    if (key >= L || (p.causal && key > row))
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
            // A row with no allowed key so far keeps m = -inf; exponentiate against 0
            // so that masked scores give exactly 0 instead of NaN.
            m_use[r] = (mx[r] == -INFINITY) ? 0.f : mx[r];
            alpha[r] = ex2(m_run[r] - m_use[r]);
            m_run[r] = mx[r];
        }

        // P = exp2(S - m) as fp16 A fragments; row sums in fp32.
        unsigned pf[kBN / 16][4];
        float rs[2] = {0.f, 0.f};
#pragma unroll
        for (int nb = 0; nb < kBN / 8; ++nb) {
            const float p0 = ex2(s[nb][0] - m_use[0]);
            const float p1 = ex2(s[nb][1] - m_use[0]);
            const float p2 = ex2(s[nb][2] - m_use[1]);
            const float p3 = ex2(s[nb][3] - m_use[1]);
            rs[0] += p0 + p1;
            rs[1] += p2 + p3;
            const int kb = nb >> 1;
            if ((nb & 1) == 0) {
                pf[kb][0] = pack_half2(p0, p1);
                pf[kb][1] = pack_half2(p2, p3);
            } else {
                pf[kb][2] = pack_half2(p0, p1);
                pf[kb][3] = pack_half2(p2, p3);
            }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r)
            l_run[r] = l_run[r] * alpha[r] + rs[r];
#pragma unroll
        for (int db = 0; db < D / 8; ++db) {
            o_acc[db][0] *= alpha[0];
            o_acc[db][1] *= alpha[0];
            o_acc[db][2] *= alpha[1];
            o_acc[db][3] *= alpha[1];
        }

        // O += P V.
#pragma unroll
        for (int kb = 0; kb < kBN / 16; ++kb) {
#pragma unroll
            for (int dp = 0; dp < D / 16; ++dp) {
                unsigned b0, b1, b2, b3;
                const int r = kb * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                const int ch = dp * 2 + (lane >> 4);
                ldsm_x4_t(b0, b1, b2, b3, v_s + swz<D>(r, ch));
                mma16816(o_acc[2 * dp], pf[kb], b0, b1);
                mma16816(o_acc[2 * dp + 1], pf[kb], b2, b3);
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();
    __syncthreads();

    // Epilogue: O / l rounded to fp16, staged through this warp's rows of sQ for 16-byte stores.
    float inv[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
        l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
        inv[r] = l_run[r] > 0.f ? 1.f / l_run[r] : 0.f;
    }
#pragma unroll
    for (int db = 0; db < D / 8; ++db) {
        const int col = (lane & 3) << 1;
        *reinterpret_cast<__half2 *>(sQ + swz<D>(wrow0 + (lane >> 2), db) + col) =
            __floats2half2_rn(o_acc[db][0] * inv[0], o_acc[db][1] * inv[0]);
        *reinterpret_cast<__half2 *>(sQ + swz<D>(wrow0 + (lane >> 2) + 8, db) + col) =
            __floats2half2_rn(o_acc[db][2] * inv[1], o_acc[db][3] * inv[1]);
    }
    __syncwarp();
    for (int c = lane; c < 16 * CPR; c += 32) {
        const int r = c / CPR, ch = c % CPR;
        const int gr = q0 + wrow0 + r;
        if (gr < N)
            *reinterpret_cast<uint4 *>(p.o + head_off + static_cast<size_t>(gr) * D + ch * 8) =
                *reinterpret_cast<const uint4 *>(sQ + swz<D>(wrow0 + r, ch));
    }
    if (p.lse && (lane & 3) == 0) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int gr = r == 0 ? row_a : row_b;
            if (gr < N)
                p.lse[static_cast<size_t>(bh) * N + gr] =
                    l_run[r] > 0.f ? (m_run[r] + log2f(l_run[r])) * kLn2 : -INFINITY;
        }
    }
}

template <int D> cudaError_t launch_d(const FwdParams &p, cudaStream_t stream)
{
    const size_t smem = static_cast<size_t>(kBM * D + 4 * kBN * D) * sizeof(__half);
    cudaError_t err = cudaFuncSetAttribute(attn_fwd_warp_mma_kernel<D>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess)
        return err;
    const int n_qtiles = (p.N + kBM - 1) / kBM;
    const long long blocks = static_cast<long long>(n_qtiles) * p.B * p.H;
    if (blocks > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    attn_fwd_warp_mma_kernel<D>
        <<<static_cast<unsigned>(blocks), kThreads, smem, stream>>>(p, n_qtiles);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_warp_mma(const FwdParams &p, cudaStream_t stream)
{
    switch (p.d) {
    case 32: return launch_d<32>(p, stream);
    case 64: return launch_d<64>(p, stream);
    case 128: return launch_d<128>(p, stream);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace attn
