// Short-sequence attention forward (N <= 256, d in {32, 64}) on the Blackwell tensor core:
// the path for many short padded sequences, e.g. a cross-encoder reranking batch (the
// "cuda-reranker" README's shape class: 50 candidates, 12 heads, head dimension 32, padded
// keys), where the work is bound by HBM traffic rather than by tensor throughput.
//
// At N <= 256 a 128-row Q tile sees at most 256 keys, so its whole score row S = Q K^T fits
// in Tensor Memory (256 fp32 columns) at once. The softmax of "Self-Attention Kernel &
// Inference Engine from Scratch" ("Online Softmax Formulation") then takes one pass over the
// row: the exponentials are taken block by block against a reference from the row's first
// block (moved, with the P already written, only when a block would leave fp16's range), and
// the accumulator is written once, by one PV product over the final P. The per-block skip of
// keys past the sequence's length (the "cuda-reranker" README's padding tile skip) is
// applied to the loads as well: K and V are fetched only up to key_lengths[b], in 32-row
// boxes, and the S product is only as wide as the allowed keys (rounded up to 16).
//
// Layout: two CTAs per SM (each holds half of Tensor Memory and about 97 KiB of shared
// memory), 6 warps each:
//   warps 0-3  softmax and epilogue of one Q tile at a time (thread r = TMEM lane r = row r)
//   warp 4     TMA producer: Q, K, V of a head into one of the CTA's head slots
//   warp 5     TMEM allocation and the single thread that issues every tcgen05.mma
// Heads are dealt to the CTAs longest-first in a snake over the grid, from the key lengths
// read on the device, so every CTA gets about the same number of score columns.
//
// TMEM (256 columns per CTA): S in columns [0, n) with n <= 256; P (fp16, two per column)
// over the first n / 2 of them; O in the last d columns. The next tile's S is issued right
// after this tile's PV product, so it overlaps the epilogue unless it reaches O's columns.
#include "attn_internal.h"
#include "sm100_ptx.cuh"

#include <cudaTypedefs.h>

#include <math.h>

namespace attn {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder(); // kernel_tcgen05.cu
cudaError_t device_sm_count(int *out);                  // kernel_tcgen05.cu

namespace {

using namespace sm100;

constexpr int kMaxN = 256;         // longest sequence this kernel takes
constexpr int kBM = 128;           // query rows per Q tile (= TMEM lanes)
constexpr int kBoxRows = 32;       // rows per TMA box
constexpr int kThreads = 192;      // 6 warps
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 256; // per CTA: two CTAs per SM share the 512 columns
constexpr int kMaxSortB = 512;      // batches sorted by key length on the device (more: natural order)
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kGuessSumMax = 32768.0f; // a block whose p sum to at most this has every p < 2^16

template <int D> struct SCfg {
    static constexpr int kRowBytes = D * 2;               // 64 B (d = 32) or 128 B: one swizzle row
    static constexpr int kTileBytes = kMaxN * kRowBytes;  // [256][D] fp16
    static constexpr int kSlots = D == 32 ? 2 : 1;        // head slots (Q, K and V of one head)
    static constexpr int kSlotBytes = 3 * kTileBytes;
    static constexpr int kBoxBytes = kBoxRows * kRowBytes;
    static constexpr uint32_t kSwizzle = D == 32 ? 4u : 2u; // descriptor layout: 64 B / 128 B swizzle
    static constexpr uint32_t kTmemO = kTmemCols - D;       // first column of the O accumulator
    static constexpr int kOffBar = kSlots * kSlotBytes;
    static constexpr int kBarBytes = 256;
    static constexpr int kOffSort = kOffBar + kBarBytes;    // key lengths, sorted order, sort keys
    static constexpr int kSmemBytes = kOffSort + 3 * kMaxSortB * 4 + 1024; // + alignment slack
    static constexpr uint32_t kIdescPV = idesc_f16_f32(kBM, D, 0, 1);
};

// Barrier block (8 bytes each).
template <int D> struct SBars {
    static constexpr int kQKFull = 0;                          // [slot] Q tile 0 and K of a head
    static constexpr int kVFull = kQKFull + SCfg<D>::kSlots;   // [slot] V of a head
    static constexpr int kSlotFree = kVFull + SCfg<D>::kSlots; // [slot] the head's last MMA is done
    static constexpr int kSFull = kSlotFree + SCfg<D>::kSlots; // S of the current tile is in TMEM
    static constexpr int kPFull = kSFull + 1;                  // P of the current tile is in TMEM
    static constexpr int kOFull = kPFull + 1;                  // O of the current tile is done
    static constexpr int kOFree = kOFull + 1;                  // O of the current tile was read
    static constexpr int kMmaDone = kOFree + 1;
    static constexpr int kQ1Full = kMmaDone + 1;               // [slot] Q tile 1 of a head
    static constexpr int kCount = kQ1Full + SCfg<D>::kSlots;
};

struct ShortArgs {
    FwdParams p;
    int n_heads;    // B * H
    int sorted;     // heads ordered by key length (1) or in batch order (0)
    unsigned int *status;
};

// The heads of this CTA: position pos of the global order (longest first) goes to CTA
// pos mod G in rounds that alternate direction, so the longest heads spread over the grid.
// A CTA takes its rounds last to first, i.e. its shortest head first: the first loads of all
// CTAs, which run before any CTA can compute, are then as small as they can be, and the
// longer heads load while the first is computed.
struct HeadCursor {
    long long round; // next round to take; -1 when done
};

__device__ __forceinline__ HeadCursor first_head(const ShortArgs &a)
{
    const long long G = gridDim.x;
    const long long c = blockIdx.x;
    long long r = (a.n_heads + G - 1) / G - 1; // last round
    while (r >= 0 && r * G + ((r & 1) ? (G - 1 - c) : c) >= a.n_heads)
        --r;
    return HeadCursor{r};
}

__device__ __forceinline__ int clamp_len(int L, int N) { return L < 0 ? 0 : (L > N ? N : L); }

__device__ __forceinline__ bool next_head(const ShortArgs &a, const int *s_len, const int *s_inv,
                                          HeadCursor &cur, int &bh, int &L)
{
    const long long G = gridDim.x;
    const long long c = blockIdx.x;
    const long long r = cur.round--;
    if (r < 0)
        return false;
    const long long pos = r * G + ((r & 1) ? (G - 1 - c) : c);
    const int H = a.p.H;
    const int rank = static_cast<int>(pos / H);
    const int h = static_cast<int>(pos - static_cast<long long>(rank) * H);
    int b = rank;
    if (a.sorted) {
        b = s_inv[rank];
        L = s_len[b];
    } else {
        L = a.p.key_lengths ? clamp_len(__ldg(a.p.key_lengths + b), a.p.N) : a.p.N;
    }
    bh = b * H + h;
    return true;
}

// Keys Q tile t attends to (the causal mask stops tile t at its last row).
__device__ __forceinline__ int tile_keys(const FwdParams &p, int L, int t)
{
    return p.causal ? min(L, (t + 1) * kBM) : L;
}

__device__ __forceinline__ uint32_t s_cols(int n_keys) { return static_cast<uint32_t>((n_keys + 15) & ~15); }

// Extreme of the 32 scores v[O .. O + 32) and a running value: three-input max (min) in a
// tree of depth 4.
template <int O, bool NEG>
__device__ __forceinline__ float chunk_ext(const uint32_t (&v)[64], float run)
{
    auto e3 = [](float a, float b, float c) { return NEG ? min3(a, b, c) : max3(a, b, c); };
    float a[8], b[4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        a[i] = e3(__uint_as_float(v[O + i]), __uint_as_float(v[O + i + 8]), __uint_as_float(v[O + i + 16]));
#pragma unroll
    for (int i = 0; i < 4; ++i)
        b[i] = e3(a[i], a[i + 4], __uint_as_float(v[O + 24 + i]));
    const float c0 = e3(b[0], b[1], __uint_as_float(v[O + 28]));
    const float c1 = e3(b[2], b[3], __uint_as_float(v[O + 29]));
    const float c2 = e3(__uint_as_float(v[O + 30]), __uint_as_float(v[O + 31]), run);
    return e3(c0, c1, c2);
}

// p_i = 2^(v_i * scale - m) for the 32 scores v[O .. O + 32), zero for entries i >= r unless
// FULL; rounded to fp16 pairs into pk and summed (fp32 pairs) into acc.
template <int O, bool FULL>
__device__ __forceinline__ void exp_chunk(const uint32_t (&v)[64], int r, uint64_t sc2, uint64_t nm2,
                                          uint64_t (&acc)[4], uint32_t (&pk)[16])
{
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(v[O + i]), __uint_as_float(v[O + i + 1])), sc2, nm2), x0, x1);
        float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
        if (!FULL) {
            p0 = i < r ? p0 : 0.f;
            p1 = i + 1 < r ? p1 : 0.f;
        }
        acc[(i >> 1) & 3] = f2_add(acc[(i >> 1) & 3], f2_pack(p0, p1));
        pk[i >> 1] = pack_f16x2(p0, p1);
    }
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;\n" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 2)
    attn_fwd_short_kernel(const ShortArgs args, const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v)
{
    using C = SCfg<D>;
    using BB = SBars<D>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    unsigned char *smem = smem_raw + (base - raw_addr);
    const uint32_t sBar = base + C::kOffBar;
    auto bar = [&](int i) -> uint32_t { return sBar + 8u * static_cast<uint32_t>(i); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffBar + 8 * BB::kCount);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *s_len = reinterpret_cast<int *>(smem + C::kOffSort);
    int *s_inv = s_len + kMaxSortB;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const FwdParams &p = args.p;
    const int N = p.N;
    const int n_qt = (N + kBM - 1) / kBM; // Q tiles per head (1 or 2)
    const uint64_t kWaitLimitNs = p.wait_limit_ns;

    // Setup that reads no input overlaps the end of the previous kernel of the stream
    // (programmatic dependent launch); inputs are read only after griddep_wait.
    if (warp == kProducerWarp && lane == 0) {
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kSlots; ++s) {
            mbar_init(bar(BB::kQKFull + s), 1);
            mbar_init(bar(BB::kVFull + s), 1);
            mbar_init(bar(BB::kSlotFree + s), 1);
            mbar_init(bar(BB::kQ1Full + s), 1);
        }
        mbar_init(bar(BB::kSFull), 1);
        mbar_init(bar(BB::kPFull), kBM);
        mbar_init(bar(BB::kOFull), 1);
        mbar_init(bar(BB::kOFree), kBM);
        mbar_init(bar(BB::kMmaDone), 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    griddep_launch_dependents();
    griddep_wait();
    // Sort keys: (length << 16) | (0xffff - index), so that "greater" means longer, or as
    // long with a smaller index. Padded to a multiple of 4 with keys smaller than any real one.
    int *s_key = s_inv + kMaxSortB;
    if (args.sorted)
        for (int b = threadIdx.x; b < ((p.B + 3) & ~3); b += kThreads) {
            const int Lb = b < p.B ? clamp_len(__ldg(p.key_lengths + b), N) : -1;
            if (b < p.B)
                s_len[b] = Lb;
            s_key[b] = Lb < 0 ? -1 : ((Lb << 16) | (0xffff - b));
        }
    // The longest-first order of the batches (rank by key length, then by index).
    if (args.sorted) {
        __syncthreads();
        const int4 *keys4 = reinterpret_cast<const int4 *>(s_key);
        const int n4 = (p.B + 3) >> 2;
        for (int b = threadIdx.x; b < p.B; b += kThreads) {
            const int kb = s_key[b];
            int rank = 0;
            for (int o = 0; o < n4; ++o) {
                const int4 q = keys4[o];
                rank += (q.x > kb) + (q.y > kb) + (q.z > kb) + (q.w > kb);
            }
            s_inv[rank] = b;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto fail = [&]() {
        *abort_flag = 1;
        *args.status = kDevStatusTimeout;
    };
    // Bounded wait of a whole warp; the outcome is made warp-uniform.
    auto warp_wait = [&](uint32_t b, uint32_t parity) -> bool {
        bool r = mbar_wait(b, parity, abort_flag, kWaitLimitNs);
        r = __all_sync(0xffffffffu, r);
        if (!r && lane == 0)
            fail();
        return r;
    };

    // The producer and MMA roles run on whole warps (converged control flow, warp-uniform
    // operands); one elected lane issues each TMA copy, tcgen05.mma and commit.
    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ TMA producer
        HeadCursor cur = first_head(args);
        int bh, L;
        uint32_t hc = 0; // heads loaded
        while (next_head(args, s_len, s_inv, cur, bh, L)) {
            if (L == 0)
                continue;
            const uint32_t slot = hc % C::kSlots;
            const uint32_t ph = (hc / C::kSlots) & 1u;
            if (!warp_wait(bar(BB::kSlotFree + slot), ph ^ 1u))
                break;
            ++hc;
            const uint32_t sQ = base + slot * C::kSlotBytes;
            const uint32_t sK = sQ + C::kTileBytes;
            const uint32_t sV = sK + C::kTileBytes;
            // Q boxes wholly past N are not loaded (their rows are never stored); K and V
            // stop at the box that holds key L - 1.
            const int q_rows = min(n_qt * kBM, N);
            const int nqb = (q_rows + kBoxRows - 1) / kBoxRows;
            const int nkv = (L + kBoxRows - 1) / kBoxRows;
            // The first score tile needs only Q tile 0 and K: they go first, under their own
            // barrier, then Q tile 1 and V (the first wave of loads is HBM-bound).
            constexpr int kTileBoxes = kBM / kBoxRows;
            const int nqb0 = nqb < kTileBoxes ? nqb : kTileBoxes;
            if (elect_one()) {
                const uint32_t qk_bar = bar(BB::kQKFull + slot);
                const uint32_t q1_bar = bar(BB::kQ1Full + slot);
                const uint32_t v_bar = bar(BB::kVFull + slot);
                mbar_arrive_expect_tx(qk_bar, (nqb0 + nkv) * C::kBoxBytes);
#pragma unroll
                for (int i = 0; i < kTileBoxes; ++i)
                    if (i < nqb0)
                        tma_load_3d(sQ + i * C::kBoxBytes, &tm_q, qk_bar, 0, i * kBoxRows, bh);
#pragma unroll
                for (int i = 0; i < kMaxN / kBoxRows; ++i)
                    if (i < nkv)
                        tma_load_3d(sK + i * C::kBoxBytes, &tm_k, qk_bar, 0, i * kBoxRows, bh);
                if (nqb > kTileBoxes) {
                    mbar_arrive_expect_tx(q1_bar, (nqb - kTileBoxes) * C::kBoxBytes);
#pragma unroll
                    for (int i = kTileBoxes; i < kMaxN / kBoxRows; ++i)
                        if (i < nqb)
                            tma_load_3d(sQ + i * C::kBoxBytes, &tm_q, q1_bar, 0, i * kBoxRows, bh);
                }
                mbar_arrive_expect_tx(v_bar, nkv * C::kBoxBytes);
#pragma unroll
                for (int i = 0; i < kMaxN / kBoxRows; ++i)
                    if (i < nkv)
                        tma_load_3d(sV + i * C::kBoxBytes, &tm_v, v_bar, 0, i * kBoxRows, bh);
            }
            __syncwarp();
        }
        // Loads still in flight land before the CTA may leave (after an abort): wait,
        // bounded by time only, for the latest fill of every slot.
        if (lane == 0)
            for (uint32_t i = hc > C::kSlots ? hc - C::kSlots : 0; i < hc; ++i) {
                mbar_wait(bar(BB::kQKFull + i % C::kSlots), (i / C::kSlots) & 1u, nullptr, kWaitLimitNs);
                if (n_qt > 1)
                    mbar_wait(bar(BB::kQ1Full + i % C::kSlots), (i / C::kSlots) & 1u, nullptr, kWaitLimitNs);
                mbar_wait(bar(BB::kVFull + i % C::kSlots), (i / C::kSlots) & 1u, nullptr, kWaitLimitNs);
            }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        bool ok = true;
        auto wait = [&](uint32_t b, uint32_t parity) -> bool {
            if (ok && !warp_wait(b, parity))
                ok = false;
            return ok;
        };
        // Shared-memory descriptors: the high word (stride byte offset = 8 rows, version,
        // swizzle) is common; the low word is (address >> 4) | (leading offset >> 4) << 16.
        constexpr uint32_t kDescHi = ((8 * C::kRowBytes) >> 4) | (1u << 14) | (C::kSwizzle << 29);
        constexpr uint32_t kLboK = (16u >> 4) << 16;                                 // K-major: unused
        constexpr uint32_t kLboV = (static_cast<uint32_t>(C::kTileBytes) >> 4) << 16; // one atom wide: unused
        auto desc = [](uint32_t lo) -> uint64_t { return (static_cast<uint64_t>(kDescHi) << 32) | lo; };
        HeadCursor cur = first_head(args);
        int bh, L;
        uint32_t hc = 0;        // heads with work
        uint32_t k = 0;         // tiles issued
        bool o_pending = false; // the last tile's O has not been seen read yet
        while (ok && next_head(args, s_len, s_inv, cur, bh, L)) {
            if (L == 0)
                continue;
            const uint32_t slot = hc % C::kSlots;
            const uint32_t ph = (hc / C::kSlots) & 1u;
            ++hc;
            const uint32_t sQ = base + slot * C::kSlotBytes;
            const uint32_t sK = sQ + C::kTileBytes;
            const uint32_t sV = sK + C::kTileBytes;
            if (!wait(bar(BB::kQKFull + slot), ph))
                break;
            for (int t = 0; t < n_qt && ok; ++t) {
                const uint32_t n_cols = s_cols(tile_keys(p, L, t));
                // S overwrites the last tile's O only when it reaches O's columns.
                if (o_pending && n_cols > C::kTmemO) {
                    if (!wait(bar(BB::kOFree), (k - 1) & 1u))
                        break;
                    o_pending = false;
                }
                if (t == 1 && !wait(bar(BB::kQ1Full + slot), ph))
                    break;
                tc_fence_after();
                const uint32_t qlo = ((sQ + t * kBM * C::kRowBytes) >> 4) | kLboK;
                const uint32_t klo = (sK >> 4) | kLboK;
                const uint32_t idesc_s = idesc_f16_f32(kBM, static_cast<int>(n_cols), 0, 0);
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        mma_ss(tmem, desc(qlo + kk * 2), desc(klo + kk * 2), idesc_s, kk > 0 ? 1u : 0u);
                    mma_commit(bar(BB::kSFull));
                }
                __syncwarp();
                // O_t = P_t V once P is in TMEM and the last tile's O has been read.
                if (!wait(bar(BB::kPFull), k & 1u))
                    break;
                if (t == 0 && !wait(bar(BB::kVFull + slot), ph))
                    break;
                if (o_pending && !wait(bar(BB::kOFree), (k - 1) & 1u))
                    break;
                tc_fence_after();
                const uint32_t vlo = (sV >> 4) | kLboV;
                const int ksteps = static_cast<int>(n_cols >> 4);
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < kMaxN / 16; ++kk)
                        if (kk < ksteps)
                            mma_ts(tmem + C::kTmemO, tmem + kk * 8, desc(vlo + kk * ((16 * C::kRowBytes) >> 4)),
                                   C::kIdescPV, kk > 0 ? 1u : 0u);
                    mma_commit(bar(BB::kOFull));
                    if (t == n_qt - 1)
                        mma_commit(bar(BB::kSlotFree + slot));
                }
                __syncwarp();
                o_pending = true;
                ++k;
            }
        }
        // Every MMA this warp issued is complete before TMEM is released (bounded by time
        // only: this wait must not give up early on an abort).
        if (elect_one())
            mma_commit(bar(BB::kMmaDone));
        __syncwarp();
        mbar_wait(bar(BB::kMmaDone), 0, nullptr, kWaitLimitNs);
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax and epilogue
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        const float scale = p.scale_log2;
        bool ok = true;
        // tcgen05.ld/st are warp-collective: every branch around them, and every decision to
        // give up, is uniform across the warp.
        auto wait_all = [&](uint32_t b, uint32_t parity) -> bool {
            bool r = mbar_wait(b, parity, abort_flag, kWaitLimitNs);
            r = __all_sync(0xffffffffu, r);
            if (!r)
                fail();
            return r;
        };
        HeadCursor cur = first_head(args);
        int bh, L;
        uint32_t k = 0;
        while (ok && next_head(args, s_len, s_inv, cur, bh, L)) {
            const size_t head_row0 = static_cast<size_t>(bh) * N;
            if (L == 0) {
                // No allowed key: O = 0 and lse = -inf for every row of the head.
                for (int t = 0; t < n_qt; ++t) {
                    const int row = t * kBM + warp * 32 + lane;
                    if (row < N) {
                        uint4 *dst = reinterpret_cast<uint4 *>(p.o + (head_row0 + row) * D);
#pragma unroll
                        for (int c = 0; c < D / 8; ++c)
                            dst[c] = make_uint4(0, 0, 0, 0);
                        if (p.lse)
                            p.lse[head_row0 + row] = -INFINITY;
                    }
                }
                continue;
            }
            for (int t = 0; t < n_qt; ++t) {
                const int n_keys = tile_keys(p, L, t);
                const int n_cols = static_cast<int>(s_cols(n_keys));
                const int n_blk = (n_cols + 63) >> 6; // 64-column blocks of S
                const int row = t * kBM + warp * 32 + lane;
                const int lim = p.causal ? min(n_keys, row + 1) : n_keys; // keys [0, lim) allowed
                const int lim_lo = __reduce_min_sync(0xffffffffu, lim);
                const int lim_hi = __reduce_max_sync(0xffffffffu, lim);
                if (!wait_all(bar(BB::kSFull), k & 1u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // One pass over the row in 64-column blocks. The exponentials use a reference
                // m_ref taken from the first block's max; it moves only when a block's max
                // exceeds it by more than 2^8 (a later block is checked through its sum, see
                // below, so every p stays inside fp16); when it moves, l and the P blocks already
                // written are rescaled by 2^(m_old - m_new). O is accumulated afterwards from the
                // final P, so the result is exact. Every decision around the warp-collective TMEM
                // accesses is made uniform across the warp.
                const bool neg = scale < 0.f;
                const float fill = neg ? INFINITY : -INFINITY;
                const uint64_t sc2 = f2_pack(scale, scale);
                float m_ref = -INFINITY;
                uint64_t acc[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    acc[i] = f2_pack(0.f, 0.f);
                for (int b = 0; b < n_blk; ++b) {
                    const int c0 = b * 64;
                    uint32_t pk[16];
                    if (c0 >= lim_hi) {
                        // no allowed key in the block for any row of the warp (causal): P = 0
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            pk[i] = 0u;
                        tmem_st16(lane_base + b * 32, pk);
                        tmem_st16(lane_base + b * 32 + 16, pk);
                        continue;
                    }
                    uint32_t v[64];
                    tmem_ld64(lane_base + c0, v);
                    const bool full = c0 + 64 <= lim_lo; // every entry allowed for every row
                    const int r = lim - c0;              // allowed entries of this block (row)
                    if (!full) {
#pragma unroll
                        for (int i = 0; i < 64; ++i)
                            v[i] = i < r ? v[i] : __float_as_uint(fill);
                    }
                    // After the first block every row has a reference (its first key is always
                    // allowed), so a later block is first exponentiated against it without a
                    // block max: when the block's sum stays <= 2^15 every p fits fp16 and the
                    // block is kept; otherwise it is redone with the block max (its scores are
                    // still in v, and P never overwrites the scores of the block being written).
                    bool guess = b > 0;
#pragma unroll 1
                    for (;;) {
                        bool any_move = false;
                        float alpha = 1.f;
                        if (!guess) {
                            const float braw = neg ? chunk_ext<32, true>(v, chunk_ext<0, true>(v, INFINITY))
                                                   : chunk_ext<32, false>(v, chunk_ext<0, false>(v, -INFINITY));
                            const float bm = braw == fill ? -INFINITY : braw * scale; // block max (log2 units)
                            const bool move = bm > m_ref + 8.f;
                            any_move = __any_sync(0xffffffffu, move);
                            if (any_move) {
                                const float m_new = move ? bm : m_ref;
                                alpha = ex2_approx(m_ref - m_new); // 0 on the first block
                                const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
                                for (int i = 0; i < 4; ++i)
                                    acc[i] = f2_fma(acc[i], a2, f2_pack(0.f, 0.f));
                                m_ref = m_new;
                            }
                        }
                        const uint64_t nm2 = f2_pack(-m_ref, -m_ref);
                        uint64_t bacc[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            bacc[i] = f2_pack(0.f, 0.f);
                        if (full)
                            exp_chunk<0, true>(v, 64, sc2, nm2, bacc, pk);
                        else
                            exp_chunk<0, false>(v, r, sc2, nm2, bacc, pk);
                        tmem_st16(lane_base + b * 32, pk);
                        if (full)
                            exp_chunk<32, true>(v, 64, sc2, nm2, bacc, pk);
                        else
                            exp_chunk<32, false>(v, r - 32, sc2, nm2, bacc, pk);
                        tmem_st16(lane_base + b * 32 + 16, pk);
                        if (guess) {
                            float s0, s1, s2, s3;
                            f2_unpack(f2_add(bacc[0], bacc[1]), s0, s1);
                            f2_unpack(f2_add(bacc[2], bacc[3]), s2, s3);
                            const float bs = (s0 + s1) + (s2 + s3);
                            if (__any_sync(0xffffffffu, !(bs <= kGuessSumMax))) {
                                tmem_wait_st(); // the redo's stores land after these
                                guess = false;
                                continue;
                            }
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            acc[i] = f2_add(acc[i], bacc[i]);
                        if (any_move && b > 0) {
                            // the P blocks written with the old reference are rescaled (fp16 pairs)
                            tmem_wait_st();
                            const uint32_t ah = pack_f16x2(alpha, alpha);
                            for (int pb = 0; pb < b; ++pb) {
                                uint32_t w[32];
                                tmem_ld32(lane_base + pb * 32, w);
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    w[i] = hmul2(w[i], ah);
                                tmem_st32(lane_base + pb * 32, w);
                            }
                        }
                        break;
                    }
                }
                float a0, a1, b0, b1;
                f2_unpack(f2_add(acc[0], acc[1]), a0, a1);
                f2_unpack(f2_add(acc[2], acc[3]), b0, b1);
                const float l = (a0 + a1) + (b0 + b1);
                const float m = m_ref;
                tmem_wait_st();
                tc_fence_before();
                // (self-test hook: withholding the first arrival makes the MMA warp's bounded
                // wait run out; never set in normal use)
                if (!(p.inject_missing_arrive && k == 0))
                    mbar_arrive(bar(BB::kPFull));
                // Epilogue: O / l -> fp16, logsumexp.
                if (!wait_all(bar(BB::kOFull), k & 1u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t ov[D];
                if constexpr (D == 32)
                    tmem_ld32(lane_base + C::kTmemO, ov);
                else
                    tmem_ld64(lane_base + C::kTmemO, ov);
                tc_fence_before();
                mbar_arrive(bar(BB::kOFree));
                ++k;
                if (row < N) {
                    const float inv = 1.f / l;
                    uint32_t h[D / 2];
#pragma unroll
                    for (int e = 0; e < D; e += 2)
                        h[e >> 1] = pack_f16x2(__uint_as_float(ov[e]) * inv, __uint_as_float(ov[e + 1]) * inv);
                    __half *orow = p.o + (head_row0 + row) * D;
                    if ((reinterpret_cast<uintptr_t>(p.o) & 31u) == 0) {
                        // whole 32-byte sectors per thread (each thread writes its own row)
#pragma unroll
                        for (int c = 0; c < D / 16; ++c)
                            st_global_v8(orow + 16 * c, h[8 * c], h[8 * c + 1], h[8 * c + 2], h[8 * c + 3],
                                         h[8 * c + 4], h[8 * c + 5], h[8 * c + 6], h[8 * c + 7]);
                    } else {
                        uint4 *dst = reinterpret_cast<uint4 *>(orow);
#pragma unroll
                        for (int c = 0; c < D / 8; ++c)
                            dst[c] = make_uint4(h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
                    }
                    if (p.lse)
                        p.lse[head_row0 + row] = (m + log2f(l)) * kLn2;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp)
        tmem_dealloc(tmem, kTmemCols);
}

// [B*H, N, D] fp16 viewed as a 3-D tensor; boxes of 32 rows x D columns with the swizzle the
// MMA descriptors expect (64-byte rows at D = 32, 128-byte rows at D = 64). Rows past N
// read as zero.
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
    using C = SCfg<D>;
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
    ShortArgs a;
    a.p = p;
    a.n_heads = BH;
    a.sorted = (p.key_lengths != nullptr && p.B <= kMaxSortB) ? 1 : 0;
    a.status = status;
    const int grid = BH < 2 * sms ? BH : 2 * sms;
    // Programmatic dependent launch: this kernel's setup may overlap the previous kernel of
    // the stream (the kernel waits for it before reading any input).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_fwd_short_kernel<D>, a, mq, mk, mv);
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
