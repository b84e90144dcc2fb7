// Warp-level building blocks of the mma.sync attention kernels: shared-memory
// swizzle, cp.async, ldmatrix, mma.sync m16n8k16 (fp16 in, fp32 accumulate), and
// WarpRows<D>, the online-softmax state of the 16 query rows one warp owns with the
// per-tile step (S = Q K^T, mask, running max and normaliser, rescale, O += P V) and
// the epilogue. The recurrence is the two-block merge of "Self-Attention Kernel &
// Inference Engine from Scratch", "Online Softmax Formulation", applied one K/V tile
// at a time.
#pragma once

#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

namespace attn {
namespace warpmma {

constexpr float kLn2 = 0.6931471805599453f;
constexpr int kTileKeys = 64; // keys per K/V tile of the warp step

// Offset (in halves) of 16-byte chunk `chunk` of row `row` in a [rows][D] tile. The
// chunk index is XOR-ed with bits of the row so that the eight rows of one ldmatrix
// phase fall into eight different bank groups. This is the same placement the TMA
// engine produces with a 128-byte swizzle for 128-byte rows (D = 64; also the low
// 128 bytes of each 256-byte row for D = 128) and with a 64-byte swizzle for 64-byte
// rows (D = 32), as long as the tile starts on a 1024-byte boundary.
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

// Online-softmax state of one warp's 16 query rows. Thread `lane` holds rows
// lane/4 and lane/4 + 8 of the warp's rows, columns 2*(lane%4) + {0, 1} of every
// 8-column block (the mma.sync accumulator layout).
template <int D> struct WarpRows {
    float o[D / 8][4];
    float m[2]; // running max, log2 units
    float l[2]; // this thread's share of the normaliser
    unsigned qf[D / 16][4];

    __device__ __forceinline__ void init()
    {
#pragma unroll
        for (int i = 0; i < D / 8; ++i)
            o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.f;
    }

    // Q fragments of rows [wrow0, wrow0 + 16) of a swizzled Q tile.
    __device__ __forceinline__ void load_q(const __half *sQ, int wrow0, int lane)
    {
#pragma unroll
        for (int kb = 0; kb < D / 16; ++kb)
            ldsm_x4(qf[kb][0], qf[kb][1], qf[kb][2], qf[kb][3],
                    sQ + swz<D>(wrow0 + (lane & 15), kb * 2 + (lane >> 4)));
    }

    // One 64-key tile: k_s / v_s point at the tile's first row (a multiple of 8 rows into
    // a swizzled buffer). kv0: index of its first key; keys >= L, and keys > row under a
    // causal mask, are excluded when need_mask is set. row_a / row_b: the last key column
    // the causal mask allows for this thread's two rows (the row index plus Nk - N).
    __device__ __forceinline__ void tile(const __half *k_s, const __half *v_s, int kv0, int L,
                                         bool causal, bool need_mask, int row_a, int row_b,
                                         float scale_log2, int lane)
    {
        float s[kTileKeys / 8][4];
#pragma unroll
        for (int nb = 0; nb < kTileKeys / 8; ++nb)
            s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.f;
        // S = Q K^T
#pragma unroll
        for (int kb = 0; kb < D / 16; ++kb) {
#pragma unroll
            for (int np = 0; np < kTileKeys / 16; ++np) {
                unsigned b0, b1, b2, b3;
                const int r = np * 16 + (lane & 7) + ((lane >> 4) << 3);
                const int ch = kb * 2 + ((lane >> 3) & 1);
                ldsm_x4(b0, b1, b2, b3, k_s + swz<D>(r, ch));
                mma16816(s[2 * np], qf[kb], b0, b1);
                mma16816(s[2 * np + 1], qf[kb], b2, b3);
            }
        }
        // scale into log2 units, mask, running max
        float mx[2] = {m[0], m[1]};
#pragma unroll
        for (int nb = 0; nb < kTileKeys / 8; ++nb) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float x = s[nb][e] * scale_log2;
                if (need_mask) {
                    const int key = kv0 + nb * 8 + ((lane & 3) << 1) + (e & 1);
                    const int row = (e < 2) ? row_a : row_b;
                    if (key >= L || (causal && key > row))
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
            alpha[r] = ex2(m[r] - m_use[r]);
            m[r] = mx[r];
        }
        // P = exp2(S - m) as fp16 A fragments; row sums in fp32
        unsigned pf[kTileKeys / 16][4];
        float rs[2] = {0.f, 0.f};
#pragma unroll
        for (int nb = 0; nb < kTileKeys / 8; ++nb) {
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
            l[r] = l[r] * alpha[r] + rs[r];
#pragma unroll
        for (int db = 0; db < D / 8; ++db) {
            o[db][0] *= alpha[0];
            o[db][1] *= alpha[0];
            o[db][2] *= alpha[1];
            o[db][3] *= alpha[1];
        }
        // O += P V
#pragma unroll
        for (int kb = 0; kb < kTileKeys / 16; ++kb) {
#pragma unroll
            for (int dp = 0; dp < D / 16; ++dp) {
                unsigned b0, b1, b2, b3;
                const int r = kb * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                const int ch = dp * 2 + (lane >> 4);
                ldsm_x4_t(b0, b1, b2, b3, v_s + swz<D>(r, ch));
                mma16816(o[2 * dp], pf[kb], b0, b1);
                mma16816(o[2 * dp + 1], pf[kb], b2, b3);
            }
        }
    }

    // Epilogue: O / l rounded to fp16 into rows [wrow0, wrow0 + 16) of the swizzled tile
    // `stage` (which the warp owns), then 16-byte stores of the rows below N to
    // `o_head` (the head's [N, D] output); lse (natural log) for the same rows.
    __device__ __forceinline__ void store(__half *stage, int wrow0, __half *o_head, float *lse_head,
                                          int row0, int N, int lane)
    {
        constexpr int CPR = D / 8;
        float inv[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
            l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
            inv[r] = l[r] > 0.f ? 1.f / l[r] : 0.f;
        }
#pragma unroll
        for (int db = 0; db < D / 8; ++db) {
            const int col = (lane & 3) << 1;
            *reinterpret_cast<__half2 *>(stage + swz<D>(wrow0 + (lane >> 2), db) + col) =
                __floats2half2_rn(o[db][0] * inv[0], o[db][1] * inv[0]);
            *reinterpret_cast<__half2 *>(stage + swz<D>(wrow0 + (lane >> 2) + 8, db) + col) =
                __floats2half2_rn(o[db][2] * inv[1], o[db][3] * inv[1]);
        }
        __syncwarp();
        for (int c = lane; c < 16 * CPR; c += 32) {
            const int r = c / CPR, ch = c % CPR;
            const int gr = row0 + r;
            if (gr < N)
                *reinterpret_cast<uint4 *>(o_head + static_cast<size_t>(gr) * D + ch * 8) =
                    *reinterpret_cast<const uint4 *>(stage + swz<D>(wrow0 + r, ch));
        }
        if (lse_head && (lane & 3) == 0) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int gr = row0 + (lane >> 2) + 8 * r;
                if (gr < N)
                    lse_head[gr] = l[r] > 0.f ? (m[r] + log2f(l[r])) * kLn2 : -INFINITY;
            }
        }
    }
};

} // namespace warpmma
} // namespace attn
