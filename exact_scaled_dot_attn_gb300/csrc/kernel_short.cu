// Short-sequence attention forward (N <= 256, d in {32, 64}): the memory-bound path
// for many short sequences, e.g. a cross-encoder reranking batch (the "cuda-reranker"
// README's shape class: B = 50 candidates, 12 heads, head dimension 32, padded keys).
//
// At these sizes a head's Q, K and V (16 KiB each at d = 32) fit on chip whole, so the
// kernel streams heads instead of tiles: a persistent grid of one 16-warp CTA per SM
// walks the heads, and while it computes one head the TMA engine already fills the
// second shared-memory stage with the next head's Q, K and V (completion on an
// mbarrier with transaction bytes). K and V are fetched only up to the head's key
// length in 64-row boxes, so padded keys are never read from HBM (the all-padding
// tile skip of the README, applied to the load as well as to the compute). Each warp
// owns 16 query rows and runs the online-softmax recurrence of "Self-Attention Kernel
// & Inference Engine from Scratch" over the resident K/V in 64-key steps (mma.sync,
// fp16 in, fp32 accumulate), stopping at its own last allowed key under a causal mask.
// The TMA swizzle (64 B rows at d = 32, 128 B rows at d = 64) is the placement the
// warp-level ldmatrix code expects, so no shared-memory bank conflicts arise.
#include "attn_internal.h"
#include "sm100_ptx.cuh"
#include "warp_mma_ops.cuh"

#include <cudaTypedefs.h>

#include <math.h>
#include <mutex>

namespace attn {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder(); // kernel_tcgen05.cu
cudaError_t device_sm_count(int *out);                  // kernel_tcgen05.cu

namespace {

using namespace warpmma;

constexpr int kMaxN = 256;   // longest sequence this kernel takes
constexpr int kBoxRows = 64; // rows per TMA box
constexpr int kWarps = kMaxN / 16;
constexpr int kThreads = kWarps * 32;

template <int D> struct ShortCfg {
    static constexpr int kTileBytes = kMaxN * D * 2; // a resident [256][D] fp16 tile
    static constexpr int kStageBytes = 3 * kTileBytes;
    static constexpr int kBoxBytes = kBoxRows * D * 2;
    static constexpr int kSmemBytes = 2 * kStageBytes + 1024 + 1024; // barriers + alignment
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_short_kernel(const FwdParams p, int n_heads, unsigned int *status,
                          const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v)
{
    using C = ShortCfg<D>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw_addr = sm100::smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    unsigned char *smem = smem_raw + (base - raw_addr);
    const uint32_t bar0 = base + 2 * C::kStageBytes; // full[0], full[1]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + 2 * C::kStageBytes + 16);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int N = p.N;

    if (tid == 0) {
        sm100::mbar_init(bar0, 1);
        sm100::mbar_init(bar0 + 8, 1);
        *abort_flag = 0;
        sm100::fence_mbarrier_init();
    }
    __syncthreads();

    auto key_length = [&](int bh) {
        int L = N;
        if (p.key_lengths) {
            L = __ldg(p.key_lengths + bh / p.H);
            L = L < 0 ? 0 : (L > N ? N : L);
        }
        return L;
    };
    // Thread 0: fetch the k-th head of this CTA into stage k % 2.
    auto issue = [&](int k) {
        const int bh = blockIdx.x + k * gridDim.x;
        if (bh >= n_heads)
            return;
        const uint32_t st = base + (k & 1) * C::kStageBytes;
        const uint32_t bar = bar0 + 8 * (k & 1);
        const int L = key_length(bh);
        const int nq = (N + kBoxRows - 1) / kBoxRows;
        const int nkv = L > 0 ? (L + kBoxRows - 1) / kBoxRows : 0;
        if (nkv == 0) {
            sm100::mbar_arrive(bar); // nothing to attend to: O = 0, no data needed
            return;
        }
        sm100::mbar_arrive_expect_tx(bar, (nq + 2 * nkv) * C::kBoxBytes);
        for (int i = 0; i < nq; ++i)
            sm100::tma_load_3d(st + i * C::kBoxBytes, &tm_q, bar, 0, i * kBoxRows, bh);
        for (int i = 0; i < nkv; ++i) {
            sm100::tma_load_3d(st + C::kTileBytes + i * C::kBoxBytes, &tm_k, bar, 0, i * kBoxRows, bh);
            sm100::tma_load_3d(st + 2 * C::kTileBytes + i * C::kBoxBytes, &tm_v, bar, 0, i * kBoxRows, bh);
        }
    };

    if (tid == 0) {
        sm100::prefetch_tensormap(&tm_q);
        sm100::prefetch_tensormap(&tm_k);
        sm100::prefetch_tensormap(&tm_v);
        issue(0);
        issue(1);
    }

    for (int k = 0;; ++k) {
        const int bh = blockIdx.x + k * gridDim.x;
        if (bh >= n_heads)
            break;
        const uint32_t bar = bar0 + 8 * (k & 1);
        bool ok = sm100::mbar_wait(bar, (k >> 1) & 1, abort_flag, p.wait_limit_ns);
        ok = __syncthreads_and(ok);
        if (!ok) {
            if (tid == 0) {
                *status = kDevStatusTimeout;
                // The two stages issued last (heads k and k + 1) may still be loading: let
                // them land, bounded by time only, before the CTA leaves.
                for (int kk = k; kk < k + 2; ++kk)
                    if (static_cast<int>(blockIdx.x) + kk * static_cast<int>(gridDim.x) < n_heads)
                        sm100::mbar_wait(bar0 + 8 * (kk & 1), (kk >> 1) & 1, nullptr, p.wait_limit_ns);
            }
            break;
        }
        __half *sQ = reinterpret_cast<__half *>(smem + (k & 1) * C::kStageBytes);
        const __half *sK = sQ + kMaxN * D;
        const __half *sV = sK + kMaxN * D;
        const int L = key_length(bh);
        const size_t head_off = static_cast<size_t>(bh) * N * D;
        const int wrow0 = warp * 16;
        if (wrow0 < N) {
            WarpRows<D> w;
            w.init();
            int kv_end = L;
            if (p.causal)
                kv_end = min(kv_end, wrow0 + 16);
            const int n_tiles = (kv_end + kTileKeys - 1) / kTileKeys;
            if (n_tiles > 0)
                w.load_q(sQ, wrow0, lane);
            const int row_a = wrow0 + (lane >> 2);
            for (int t = 0; t < n_tiles; ++t) {
                const int kv0 = t * kTileKeys;
                const bool need_mask = (kv0 + kTileKeys > L) || (p.causal && kv0 + kTileKeys - 1 > wrow0);
                w.tile(sK + kv0 * D, sV + kv0 * D, kv0, L, p.causal != 0, need_mask, row_a, row_a + 8,
                       p.scale_log2, lane);
            }
            w.store(sQ, wrow0, p.o + head_off, p.lse ? p.lse + static_cast<size_t>(bh) * N : nullptr,
                    wrow0, N, lane);
        }
        __syncthreads(); // every warp is done with this stage
        if (tid == 0) {
            // The stage was read (and its Q rows rewritten) through the generic proxy;
            // order that before the TMA engine writes the stage again.
            asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
            issue(k + 2);
        }
    }
}

// [B*H, N, D] fp16 viewed as a 3-D tensor; boxes of 64 rows x D columns; the swizzle
// matches swz<D>: 64-byte for D = 32, 128-byte for D = 64. Rows past N read as zero.
bool encode_short_map(CUtensorMap *m, const void *ptr, int BH, int N, int D)
{
    auto enc = tensor_map_encoder();
    if (!enc)
        return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                             static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(D) * 2};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(D), static_cast<cuuint32_t>(kBoxRows), 1};
    cuuint32_t es[3] = {1, 1, 1};
    const CUtensorMapSwizzle sw = D == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D> cudaError_t launch_d(const FwdParams &p, cudaStream_t stream, unsigned int *status)
{
    using C = ShortCfg<D>;
    const int BH = p.B * p.H;
    CUtensorMap mq, mk, mv;
    if (!encode_short_map(&mq, p.q, BH, p.N, D) || !encode_short_map(&mk, p.k, BH, p.N, D) ||
        !encode_short_map(&mv, p.v, BH, p.N, D))
        return cudaErrorInvalidValue;
    int sms = 0;
    cudaError_t err = device_sm_count(&sms);
    if (err != cudaSuccess)
        return err;
    err = cudaFuncSetAttribute(attn_fwd_short_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               C::kSmemBytes);
    if (err != cudaSuccess)
        return err;
    const int grid = BH < sms ? BH : sms;
    attn_fwd_short_kernel<D><<<grid, kThreads, C::kSmemBytes, stream>>>(p, BH, status, mq, mk, mv);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_short(const FwdParams &p, cudaStream_t stream, unsigned int *status)
{
    if (p.N > kMaxN)
        return cudaErrorInvalidValue;
    switch (p.d) {
    case 32: return launch_d<32>(p, stream, status);
    case 64: return launch_d<64>(p, stream, status);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace attn
