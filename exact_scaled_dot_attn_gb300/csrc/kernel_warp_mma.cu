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
// Cross-attention and grouped-query attention: the K/V rows come from the query
// head's key/value head (Nk keys), and the causal diagonal moves by Nk - N.
//
// This kernel serves every head dimension and length but is on no automatic path: the
// tcgen05 kernels are faster at every measured shape (the short-sequence kernel for d = 32
// with N <= 256, the tiled kernel elsewhere). It is kept as an independent second
// implementation that is selected explicitly (ATTN_PATH_WARP_MMA) and run by the parity tests.
#include "attn_internal.h"

#include <math.h>

#include "warp_mma_ops.cuh"

namespace attn {
namespace {

using namespace warpmma;

constexpr int kBM = 64; // query rows per CTA: 4 warps x 16 rows
constexpr int kBN = kTileKeys; // keys per K/V tile
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;

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
    const int N = p.N, Nk = p.Nk;
    const int diag = Nk - N; // causal: query i sees keys j <= i + diag
    const int q0 = qt * kBM;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    int L = Nk;
    if (p.key_lengths) {
        L = p.key_lengths[b];
        L = L < 0 ? 0 : (L > Nk ? Nk : L);
    }
    int kv_end = L;
    if (p.causal && !p.qrows) // (packed query groups: every tile sees all keys up to L)
        kv_end = max(0, min(kv_end, q0 + kBM + diag));
    // packed query groups: row r is query r % qrows, whose diagonal is at Nk - qrows
    const int qdiag = p.qrows ? Nk - p.qrows : diag;
    const int n_tiles = (kv_end + kBN - 1) / kBN;

    const size_t head_off = static_cast<size_t>(bh) * N * D;
    const int kvh = b * p.Hkv + (bh - b * p.H) / (p.H / p.Hkv);
    const size_t kv_off = static_cast<size_t>(kvh) * Nk * D;
    const __half *gQ = p.q + head_off;
    const __half *gK = p.k + kv_off;
    const __half *gV = p.v + kv_off;

    // Rows [r0, r0 + rows) of one head into a swizzled tile; rows >= n are zero-filled.
    auto load_tile = [&](__half *s, const __half *g, int r0, int rows, int n) {
        for (int c = tid; c < rows * CPR; c += kThreads) {
            const int r = c / CPR, ch = c % CPR;
            const int gr = r0 + r;
            const bool ok = gr < n;
            const __half *src = g + static_cast<size_t>(ok ? gr : 0) * D + ch * 8;
            cp_async16(s + swz<D>(r, ch), src, ok);
        }
    };

    load_tile(sQ, gQ, q0, kBM, N);
    if (n_tiles > 0) {
        load_tile(sK, gK, 0, kBN, Nk);
        load_tile(sV, gV, 0, kBN, Nk);
    }
    cp_async_commit();

    WarpRows<D> w;
    w.init();
    const int wrow0 = warp * 16;
    const int row_a = q0 + wrow0 + (lane >> 2);
    const int row_b = row_a + 8;

    for (int t = 0; t < n_tiles; ++t) {
        const int st = t & 1;
        if (t + 1 < n_tiles) {
            load_tile(sK + (st ^ 1) * kBN * D, gK, (t + 1) * kBN, kBN, Nk);
            load_tile(sV + (st ^ 1) * kBN * D, gV, (t + 1) * kBN, kBN, Nk);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        if (t == 0)
            w.load_q(sQ, wrow0, lane);
        const int kv0 = t * kBN;
        const bool need_mask = (kv0 + kBN > L) ||
                               (p.causal && kv0 + kBN - 1 > (p.qrows ? qdiag : q0 + wrow0 + diag));
        // the masks compare keys with the diagonal column of each row: row + diag
        const int da = (p.qrows ? row_a % p.qrows : row_a) + qdiag;
        const int db = (p.qrows ? row_b % p.qrows : row_b) + qdiag;
        w.tile(sK + st * kBN * D, sV + st * kBN * D, kv0, L, p.causal != 0, need_mask, da, db,
               p.scale_log2, lane);
        __syncthreads();
    }
    cp_async_wait<0>();
    __syncthreads();

    // Epilogue through this warp's rows of sQ.
    w.store(sQ, wrow0, p.o + head_off, p.lse ? p.lse + static_cast<size_t>(bh) * N : nullptr,
            q0 + wrow0, N, lane);
}

template <int D> cudaError_t launch_d(const FwdParams &p, cudaStream_t stream)
{
    if (p.Hkv < 1 || p.H % p.Hkv != 0)
        return cudaErrorInvalidValue;
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
