// TMA + tcgen05/TMEM attention forward for sm_103a (head dimension 32, 64 or 128).
//
// The tiled online-softmax recurrence of "Self-Attention Kernel & Inference
// Engine from Scratch" ("Online Softmax Formulation", "CUDA Kernel Structure"),
// laid out for the Blackwell tensor core:
//
//   work unit   (batch*head, pair of 128-row Q tiles), in a host-built order: heads are
//               taken in blocks whose K/V fit comfortably in L2, and inside a block the
//               units go heaviest-first (last query rows first under a causal mask). With
//               at least three units per SM the grid has one CTA per unit and running CTAs
//               take over the units of CTAs that have not started (cluster launch
//               control), so faster CTAs take more units; otherwise a persistent grid of
//               one CTA per SM walks host-built largest-first lists.
//               Cross-attention and grouped-query attention (the README's "natural
//               extensions"): Q tiles are rows of a query head, K/V tiles come from
//               its key/value head, and the causal diagonal moves by Nk - N.
//   warp 8      TMA producer: Q0/Q1 once per unit, then K_j and V_j through a ring of
//               shared-memory stages (full/empty mbarriers with transaction counts).
//               K/V tiles past the causal diagonal or past key_lengths[b] are never
//               loaded (the block skip of "Engineering Decisions & Trade-offs" and the
//               padding tile skip of the "cuda-reranker" README).
//   warp 9      allocates TMEM and issues every tcgen05.mma from one thread:
//               S_t = Q_t K_j^T (fp16 x fp16 -> fp32 in TMEM) and O_t += P_t V_j with
//               P_t read from TMEM; completion is signalled with tcgen05.commit.
//   warps 0-3   softmax warpgroup for Q tile 0, warps 4-7 for Q tile 1: thread r owns
//               TMEM lane r = query row r. Per K/V tile it reads the S row (one TMEM
//               load of 128 columns), scales,
//               masks, updates the running max m and normaliser l with exp2, and writes
//               P (fp16) into TMEM over S. The accumulator O is rescaled only when the
//               row max grows by more than 2^8 over the reference used so far (lazy
//               correction: O and l always share one reference, so the result is exact).
//               At the end of the unit it divides O by l, rounds to fp16, stores O and
//               the logsumexp.
//
// TMEM columns: S0 [0,128) S1 [128,256), then the O accumulators from column 256 (O_t of
// buffer b at 256 + (2b + t) d: one buffer per tile at d = 128 and d = 64, two at d = 32).
// P_t is packed 16-bit in the first 64 columns of S_t (fp32 P of the tf32 kind fills all 128),
// except at d = 64 (16-bit), where it has its own columns [384, 448) and [448, 512). Every
// mbarrier wait is bounded; a wait that runs
// out sets the abort flag and the device status word and the CTA unwinds.
#include "attn_internal.h"
#include "sm100_ptx.cuh"

#include <cudaTypedefs.h>

#include <math.h>
#include <string.h>
#include <algorithm>
#include <map>
#include <memory>
#include <mutex>
#include <queue>
#include <tuple>
#include <vector>

namespace attn {

// cuTensorMapEncodeTiled, looked up once through the runtime (no link against libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}


namespace {
constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices];
std::mutex g_sm_mutex;

cudaError_t sm_count_locked(int *out)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_sm_mutex);
    if (!g_sm_count[dev]) {
        err = cudaDeviceGetAttribute(&g_sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
        if (err != cudaSuccess)
            return err;
    }
    *out = g_sm_count[dev];
    return cudaSuccess;
}

} // namespace

// Multiprocessor count of the current device (cached per device).
cudaError_t device_sm_count(int *out) { return sm_count_locked(out); }

namespace {

using namespace sm100;

constexpr int kBM = 128;      // query rows per Q tile
constexpr int kBN = 128;      // keys per K/V tile
constexpr int kThreads = 384; // 12 warps: softmax warpgroups 0 and 1, control warpgroup 2
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
// Register split after launch: the softmax warpgroups hold a 128-column S row in
// registers, the control warpgroup (TMA, MMA and two idle warps) needs few; at d = 128
// the unrolled MMA issue of the control warpgroup needs more than at d <= 64. The pool is
// what the CTA launched with (threads x registers per thread); the host checks that
// 8 * 32 * softmax + 4 * 32 * control fits in it before launching.
template <int D> struct RegSplit {
    static constexpr uint32_t kSoftmax = 208;
    static constexpr uint32_t kControl = D == 128 ? 88 : 72;
    static constexpr int kPoolNeeded = 8 * 32 * kSoftmax + 4 * 32 * kControl;
};
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f; // lazy-correction threshold (log2 units)

// Element kinds of Q, K, V and O: fp16 and bf16 run tcgen05.mma kind::f16; fp32 inputs run
// kind::tf32 (the tensor core reads 10 fraction bits of each fp32 value).
constexpr int kKindF16 = 0;
constexpr int kKindBF16 = 1;
constexpr int kKindTF32 = 2;
template <int KIND> __host__ __device__ constexpr int elem_bytes() { return KIND == kKindTF32 ? 4 : 2; }

// Tile geometry for head dimension D and ES-byte elements. A TMA box row is one swizzle row
// (64 bytes for fp16 at d = 32, 128 bytes otherwise); fp32 at d = 32 has the byte geometry of
// fp16 at d = 64.
template <int D, int ES = 2> struct Cfg {
    static constexpr int kBoxCols = D * ES < 128 ? D : 128 / ES; // elements per TMA box row
    static constexpr int kRowBytes = kBoxCols * ES;     // 64 B or 128 B
    static constexpr int kBoxBytes = kBM * kRowBytes;  // one 128-row box
    static constexpr int kTileBytes = kBM * D * ES;    // a 128 x D tile (D / kBoxCols boxes)
    static constexpr uint32_t kSwizzle = kRowBytes < 128 ? 4u : 2u; // descriptor layout: 64 B / 128 B swizzle
    static constexpr int kKStep = 32 / ES;             // K elements per MMA instruction (32 bytes)
    static constexpr int kQStages = kTileBytes >= 32768 ? 1 : 2; // Q0/Q1 buffers (2: next unit prefetched)
    // fp32 (tf32) tiles: the PV product needs V K-major (tf32 operands cannot be MN-major), so
    // each V tile is transposed into one of kVTStages V^T buffers, taking two ring stages' room.
    static constexpr int kVTStages = ES == 4 ? 2 : 0;
    static constexpr int kStages = ES == 4 ? 7 : (kTileBytes >= 32768 ? 5 : (kTileBytes >= 16384 ? 9 : 16)); // K/V ring
    static constexpr uint32_t kTmemS0 = 0, kTmemS1 = 128;
    // Separate P (d = 64, 16-bit elements): P_t gets its own 64 TMEM columns instead of the
    // first half of S_t, so S_t(j+1) is issued as soon as the softmax has read S_t(j), before
    // O_t += P_t(j) V_j; the softmax of the next step then finds its scores ready. The columns
    // come from the second O buffer (one O buffer per tile here).
    static constexpr bool kSepP = D == 64 && ES == 2;
    static constexpr uint32_t kTmemP0 = 384, kTmemP1 = 448;
    // O accumulators: two per Q tile when they fit (d <= 64), so that a unit's epilogue
    // can read one while the next unit's PV products accumulate into the other.
    static constexpr int kOBufs = (D <= 64 && !kSepP) ? 2 : 1;
    static constexpr uint32_t kTmemCols = 512;
    __host__ __device__ static constexpr uint32_t tmem_o(int t, int b)
    {
        return 256u + static_cast<uint32_t>((b * 2 + t) * D);
    }
    static constexpr int kOffQ = 0;
    static constexpr int kOffKV = kQStages * 2 * kTileBytes;
    static constexpr int kOffVT = kOffKV + kStages * kTileBytes;
    static constexpr int kOffBar = kOffVT + kVTStages * kTileBytes;
    static constexpr int kSmemBytes = kOffBar + 1024 + 1024; // barriers + alignment slack
};

struct TcArgs {
    FwdParams p;
    int n_pairs; // ceil(N / 256)
    int n_units; // n_pairs * B * H * n_splits
    int head_block; // heads per L2 block of the unit order
    int n_splits;   // key ranges per (batch*head, Q tile pair); 1 outside split-KV
    // Balanced split-KV (bal_chunks > 0): the K/V tiles of all (batch*head, pair) units, bal_nfull
    // per pair, laid end to end and cut into bal_chunks equal runs (one per CTA); range s of a
    // pair is its part of the s-th run that touches it (empty when there is none).
    int bal_chunks;
    int bal_nfull;
    float *opart;   // split-KV partial outputs: [split][B*H*N][D] fp32, O / l of the range
    float *lpart;   // split-KV partial logsumexp: [split][B*H*N] fp32 (-inf: no key in the range)
    unsigned int *status;
    // 1: one CTA per unit, CTA c running unit unit[c] of the schedule table (unit c when the
    // table is not used); a running CTA takes over the units of CTAs that have not started
    // (cluster launch control), so the CTAs that finish first take more units. 0: a persistent
    // grid walks the table's per-CTA lists.
    int dynamic;
};

struct Unit {
    int bh, b, q0, L;
    int kvh;        // key/value head (batch * Hkv + h / (H / Hkv))
    int n_kv;       // K/V tiles loaded for the unit (the larger of the two tile counts)
    int n_kv_t[2];  // K/V tiles Q tile t attends to (0 when the tile lies past N)
    int j0;         // first K/V tile of the unit's key range (split-KV; 0 otherwise)
    int split;      // index of that range
};

// Schedule table computed on the host. Static schedule: CTA c processes the units
// unit[off[c] .. off[c+1]) in that order (largest-first assignment to the least loaded CTA,
// head block by head block); when `use` is 0 the CTAs walk the unit order in a snake instead.
// Dynamic schedule (TcArgs::dynamic): CTA id c runs unit unit[c] (off is unused); when `use`
// is 0, unit c.
constexpr int kMaxCtas = 256;
constexpr int kMaxSchedUnits = 4096;
struct SchedTable {
    int use;
    uint16_t off[kMaxCtas + 1];
    uint16_t unit[kMaxSchedUnits];
};

__device__ __forceinline__ Unit decode_unit(const TcArgs &a, int u)
{
    const int BH = a.p.B * a.p.H;
    Unit U;
    const int S = a.n_splits;
    const int per_block = a.head_block * a.n_pairs * S;
    const int blk = u / per_block;
    const int ws = u - blk * per_block;
    const int split = ws % S; // the key ranges of one (head, pair) are adjacent in the order
    const int w = ws / S;
    const int h0 = blk * a.head_block;
    const int hb = min(a.head_block, BH - h0);
    const int pair = a.n_pairs - 1 - w / hb; // the last query rows carry the most causal work
    U.bh = h0 + w % hb;
    U.b = U.bh / a.p.H;
    U.kvh = U.b * a.p.Hkv + (U.bh - U.b * a.p.H) / (a.p.H / a.p.Hkv);
    U.q0 = pair * 2 * kBM;
    int L = a.p.Nk;
    if (a.p.key_lengths) {
        L = __ldg(a.p.key_lengths + U.b);
        L = L < 0 ? 0 : (L > a.p.Nk ? a.p.Nk : L);
    }
    U.L = L;
    int kv_end0 = L, kv_end1 = L;
    // (packed query groups: every 128-row tile holds a last query of some head, so no K/V
    // tile is skipped by the causal mask)
    if (a.p.causal && !a.p.qrows) {
        // Q tile 0 stops at its own diagonal (query i sees keys j <= i + Nk - N)
        const int off = a.p.Nk - a.p.N;
        kv_end0 = max(0, min(L, U.q0 + kBM + off));
        kv_end1 = max(0, min(L, U.q0 + 2 * kBM + off));
    }
    const int full0 = (kv_end0 + kBN - 1) / kBN;
    const int full1 = U.q0 + kBM < a.p.N ? (kv_end1 + kBN - 1) / kBN : 0;
    const int n_full = max(full0, full1);
    // Key range of this split: K/V tiles [j0, j1) of the pair's n_full tiles.
    int j0 = split * n_full / S;
    int j1 = (split + 1) * n_full / S;
    if (a.bal_chunks > 0) {
        // run c covers tiles [c T / G, (c + 1) T / G) of the T laid end to end; the pair (w-th in
        // the unit order, one head block) starts at tile w * nf, inside run c0
        const long long nf = a.bal_nfull, G = a.bal_chunks;
        const long long T = static_cast<long long>(BH) * a.n_pairs * nf;
        const long long t0 = static_cast<long long>(w) * nf;
        const long long c = ((t0 + 1) * G - 1) / T + split;
        const long long lo = c * T / G, hi = (c + 1) * T / G;
        const long long a0 = lo > t0 ? lo : t0, a1 = hi < t0 + nf ? hi : t0 + nf;
        j0 = c < G && a0 < a1 ? static_cast<int>(a0 - t0) : 0;
        j1 = c < G && a0 < a1 ? static_cast<int>(a1 - t0) : 0;
        j1 = min(j1, n_full); // past the keys this pair really has (key lengths)
        j0 = min(j0, j1);
    }
    U.j0 = j0;
    U.split = split;
    U.n_kv_t[0] = max(0, min(j1, full0) - j0);
    U.n_kv_t[1] = max(0, min(j1, full1) - j0);
    U.n_kv = j1 - j0;
    return U;
}

// K/V tile count of Q tile t, without indexing a local array by a runtime value.
__device__ __forceinline__ int kv_tiles(const Unit &U, int t) { return t ? U.n_kv_t[1] : U.n_kv_t[0]; }

// Unit of round r for CTA c: consecutive rounds walk the CTAs in opposite directions.
__device__ __forceinline__ int unit_at(int r, int c, int G)
{
    return r * G + ((r & 1) ? (G - 1 - c) : c);
}

// The sequence of units of one CTA; every role of the CTA walks the same sequence.
struct UnitCursor {
    int i, end, r;
};
__device__ __forceinline__ UnitCursor first_unit(const SchedTable &s)
{
    UnitCursor c;
    c.i = s.use ? s.off[blockIdx.x] : 0;
    c.end = s.use ? s.off[blockIdx.x + 1] : 0;
    c.r = 0;
    return c;
}
__device__ __forceinline__ bool next_unit(const TcArgs &a, const SchedTable &s, UnitCursor &c, int &u)
{
    if (s.use) {
        if (c.i >= c.end)
            return false;
        u = s.unit[c.i++];
        return true;
    }
    u = unit_at(c.r++, blockIdx.x, gridDim.x);
    return u < a.n_units;
}

// The CTA's units, decoded one ahead: taking a unit starts decoding the following one,
// so its key-length load is in flight while the taken unit is processed.
struct UnitStream {
    UnitCursor cur;
    bool has;
    Unit next;
    uint32_t k; // dynamic schedule: units taken from the shared ring
};
__device__ __forceinline__ void stream_init(UnitStream &st, const TcArgs &a, const SchedTable &s)
{
    st.k = 0;
    if (a.dynamic) {
        st.has = true; // every unit, the first included, comes from the ring
        return;
    }
    st.cur = first_unit(s);
    int u;
    st.has = next_unit(a, s, st.cur, u);
    if (st.has)
        st.next = decode_unit(a, u);
}
__device__ __forceinline__ bool stream_take(UnitStream &st, const TcArgs &a, const SchedTable &s, Unit &U)
{
    if (!st.has)
        return false;
    U = st.next;
    int u;
    st.has = next_unit(a, s, st.cur, u);
    if (st.has)
        st.next = decode_unit(a, u);
    return true;
}

// Barrier block layout (8 bytes each).
template <int D, int ES = 2> struct Bars {
    static constexpr int kQFull = 0;                                  // [kQStages]
    static constexpr int kQEmpty = kQFull + Cfg<D, ES>::kQStages;     // [kQStages]
    static constexpr int kKVFull = kQEmpty + Cfg<D, ES>::kQStages;
    static constexpr int kKVEmpty = kKVFull + Cfg<D, ES>::kStages;
    static constexpr int kSFull = kKVEmpty + Cfg<D, ES>::kStages; // [2]
    static constexpr int kPFull = kSFull + 2;                 // [2]
    static constexpr int kOReady = kPFull + 2;                // [tile * 2 + O buffer]
    static constexpr int kOEmpty = kOReady + 4;               // [tile * 2 + O buffer]
    static constexpr int kMmaDone = kOEmpty + 4;
    // tf32 only: V tile landed (MMA warp -> transposer warps), V^T written, V^T buffer free
    static constexpr int kVReady = kMmaDone + 1;  // [2]
    static constexpr int kVTFull = kVReady + 2;   // [2]
    static constexpr int kVTEmpty = kVTFull + 2;  // [2]
    // separate P only: the softmax of tile t has read S_t (the next S_t may be written)
    static constexpr int kSFree = kVTEmpty + 2;   // [2]
    // dynamic schedule: the ring of decoded units (producer -> other roles) and the answer of
    // the cluster launch control request in flight
    static constexpr int kUnitFull = kSFree + 2;  // [kUnitSlots]
    static constexpr int kUnitEmpty = kUnitFull + 4;
    static constexpr int kClc = kUnitEmpty + 4;
    static constexpr int kCount = kClc + 1;
    // byte offsets from the start of the barrier block (which has 1 KB)
    static constexpr int kClcResp = 640;  // 16-byte answer
    static constexpr int kUnitRing = 656; // kUnitSlots units
    static_assert(8 * kCount + 8 <= kClcResp, "barrier block overflow");
};
constexpr int kUnitSlots = 4;
static_assert(Bars<128>::kUnitRing + kUnitSlots * static_cast<int>(sizeof(Unit)) <= 1024, "unit ring overflow");

// Column chunks of the S row: the allowed columns of a row are a prefix e < lim (key
// padding and the causal diagonal both cut a row at one column), so every 32-column chunk
// is fully allowed, fully masked, or the single boundary chunk. Only the boundary chunk
// pays for per-element masking; fully masked chunks cost nothing.
constexpr int kChunkCols = 32;

// Max (min when `neg`) of the raw scores of one fully allowed chunk: three-input max
// over eight independent chains.
template <bool NEG>
__device__ __forceinline__ float chunk_extreme(const uint32_t (&sv)[kBN], int c)
{
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        acc[i] = NEG ? fminf(__uint_as_float(sv[c * 32 + i]), __uint_as_float(sv[c * 32 + 8 + i]))
                     : fmaxf(__uint_as_float(sv[c * 32 + i]), __uint_as_float(sv[c * 32 + 8 + i]));
#pragma unroll
    for (int i = 0; i < 8; ++i)
        acc[i] = NEG ? min3(acc[i], __uint_as_float(sv[c * 32 + 16 + i]), __uint_as_float(sv[c * 32 + 24 + i]))
                     : max3(acc[i], __uint_as_float(sv[c * 32 + 16 + i]), __uint_as_float(sv[c * 32 + 24 + i]));
    return NEG ? min3(min3(acc[0], acc[1], acc[2]), min3(acc[3], acc[4], acc[5]), fminf(acc[6], acc[7]))
               : max3(max3(acc[0], acc[1], acc[2]), max3(acc[3], acc[4], acc[5]), fmaxf(acc[6], acc[7]));
}

// Row max of the scaled scores over a fully allowed row: the extreme of the raw scores
// (the min when the scale is negative) by three-input max over eight independent
// chains, scaled once.
__device__ __forceinline__ float row_max_full(const uint32_t (&sv)[kBN], float scale)
{
    float acc[8];
    if (scale >= 0.f) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            acc[i] = fmaxf(__uint_as_float(sv[i]), __uint_as_float(sv[i + 8]));
#pragma unroll
        for (int e = 16; e < kBN; e += 16)
#pragma unroll
            for (int i = 0; i < 8; ++i)
                acc[i] = max3(acc[i], __uint_as_float(sv[e + i]), __uint_as_float(sv[e + 8 + i]));
        return max3(max3(acc[0], acc[1], acc[2]), max3(acc[3], acc[4], acc[5]), fmaxf(acc[6], acc[7])) * scale;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
        acc[i] = fminf(__uint_as_float(sv[i]), __uint_as_float(sv[i + 8]));
#pragma unroll
    for (int e = 16; e < kBN; e += 16)
#pragma unroll
        for (int i = 0; i < 8; ++i)
            acc[i] = min3(acc[i], __uint_as_float(sv[e + i]), __uint_as_float(sv[e + 8 + i]));
    return min3(min3(acc[0], acc[1], acc[2]), min3(acc[3], acc[4], acc[5]), fminf(acc[6], acc[7])) * scale;
}

// p_e = 2^(S_e * scale - m) over a fully allowed row, stored to TMEM at tP: rounded to
// 16-bit pairs (fp16 or bf16) in two halves of 32 columns, or (tf32) as fp32 in 128 columns
// over the row's own scores; returns sum_e p_e in fp32 (f32x2 arithmetic).
template <int KIND>
__device__ __forceinline__ float exp_pack_full(uint32_t (&sv)[kBN], float scale, float neg_m,
                                               uint32_t tP)
{
    const uint64_t sc2 = f2_pack(scale, scale);
    const uint64_t nm2 = f2_pack(neg_m, neg_m);
    uint64_t acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        acc[i] = f2_pack(0.f, 0.f);
    if constexpr (KIND == kKindTF32) {
        // each p replaces its own score in sv (no second 128-value array)
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c) {
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                const int e = c * 32 + i;
                float x0, x1;
                f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), sc2, nm2), x0, x1);
                const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                acc[(i >> 1) & 3] = f2_add(acc[(i >> 1) & 3], f2_pack(p0, p1));
                sv[e] = __float_as_uint(p0);
                sv[e + 1] = __float_as_uint(p1);
            }
            tmem_st32(tP + c * 32, *reinterpret_cast<const uint32_t(*)[32]>(&sv[c * 32]));
        }
        float a0, a1, b0, b1;
        f2_unpack(f2_add(acc[0], acc[1]), a0, a1);
        f2_unpack(f2_add(acc[2], acc[3]), b0, b1);
        return (a0 + a1) + (b0 + b1);
    } else {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t pk[32];
#pragma unroll
            for (int i = 0; i < 64; i += 2) {
                const int e = half * 64 + i;
                float x0, x1;
                f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), sc2, nm2), x0, x1);
                const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                acc[(i >> 1) & 3] = f2_add(acc[(i >> 1) & 3], f2_pack(p0, p1));
                pk[i >> 1] = pack2<KIND == kKindBF16>(p0, p1);
            }
            tmem_st32(tP + half * 32, pk);
        }
        float a0, a1, b0, b1;
        f2_unpack(f2_add(acc[0], acc[1]), a0, a1);
        f2_unpack(f2_add(acc[2], acc[3]), b0, b1);
        return (a0 + a1) + (b0 + b1);
    }
}

// Row max of the scaled scores x_e = S_e * scale over the allowed columns e < lim
// (lim >= 128: the whole row). Fully allowed chunks take the extreme of the raw scores
// (the min when the scale is negative) and scale it once.
__device__ __forceinline__ float row_max(const uint32_t (&sv)[kBN], float scale, int lim)
{
    float m = -INFINITY;
#pragma unroll
    for (int c = 0; c < kBN / kChunkCols; ++c) {
        if (lim >= (c + 1) * kChunkCols) {
            const float r = scale >= 0.f ? chunk_extreme<false>(sv, c) : chunk_extreme<true>(sv, c);
            m = fmaxf(m, r * scale);
        } else if (lim > c * kChunkCols) {
#pragma unroll
            for (int i = 0; i < kChunkCols; ++i) {
                const int e = c * kChunkCols + i;
                const float x = e < lim ? __uint_as_float(sv[e]) * scale : -INFINITY;
                m = fmaxf(m, x);
            }
        }
    }
    return m;
}

// p_e = 2^(S_e * scale - m) for the allowed columns e < lim, 0 elsewhere, stored to TMEM at
// tP as exp_pack_full stores it (16-bit pairs in two halves of 32 columns, so only half of the
// packed row is held in registers at a time, or fp32 for tf32); returns sum_e p_e in fp32.
// Pairs of lanes use f32x2 arithmetic; fully masked chunks store zeros without evaluating any
// exponential.
template <int KIND>
__device__ __forceinline__ float exp_pack(uint32_t (&sv)[kBN], float scale, float neg_m, int lim,
                                          uint32_t tP)
{
    const uint64_t sc2 = f2_pack(scale, scale);
    const uint64_t nm2 = f2_pack(neg_m, neg_m);
    uint64_t acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        acc[i] = f2_pack(0.f, 0.f);
    if constexpr (KIND == kKindTF32) {
        // each p replaces its own score in sv (no second 128-value array)
#pragma unroll
        for (int c = 0; c < kBN / kChunkCols; ++c) {
            uint32_t(&pv)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[c * kChunkCols]);
            if (lim >= (c + 1) * kChunkCols) {
#pragma unroll
                for (int i = 0; i < kChunkCols; i += 2) {
                    const int e = c * kChunkCols + i;
                    float x0, x1;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), sc2, nm2), x0, x1);
                    const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                    acc[(i >> 1) & 3] = f2_add(acc[(i >> 1) & 3], f2_pack(p0, p1));
                    pv[i] = __float_as_uint(p0);
                    pv[i + 1] = __float_as_uint(p1);
                }
            } else if (lim > c * kChunkCols) {
#pragma unroll
                for (int i = 0; i < kChunkCols; i += 2) {
                    const int e = c * kChunkCols + i;
                    float x0, x1;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), sc2, nm2), x0, x1);
                    const float p0 = e < lim ? ex2_approx(x0) : 0.f;
                    const float p1 = e + 1 < lim ? ex2_approx(x1) : 0.f;
                    acc[(i >> 1) & 3] = f2_add(acc[(i >> 1) & 3], f2_pack(p0, p1));
                    pv[i] = __float_as_uint(p0);
                    pv[i + 1] = __float_as_uint(p1);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    pv[i] = 0u;
            }
            tmem_st32(tP + c * 32, pv);
        }
        float a0, a1, b0, b1;
        f2_unpack(f2_add(acc[0], acc[1]), a0, a1);
        f2_unpack(f2_add(acc[2], acc[3]), b0, b1);
        return (a0 + a1) + (b0 + b1);
    } else {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t pk[32];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int c = half * 2 + cc;
                if (lim >= (c + 1) * kChunkCols) {
#pragma unroll
                    for (int i = 0; i < kChunkCols; i += 2) {
                        const int e = c * kChunkCols + i;
                        float x0, x1;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), sc2, nm2), x0, x1);
                        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                        acc[(i >> 1) & 3] = f2_add(acc[(i >> 1) & 3], f2_pack(p0, p1));
                        pk[cc * 16 + (i >> 1)] = pack2<KIND == kKindBF16>(p0, p1);
                    }
                } else if (lim > c * kChunkCols) {
#pragma unroll
                    for (int i = 0; i < kChunkCols; i += 2) {
                        const int e = c * kChunkCols + i;
                        float x0, x1;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), sc2, nm2), x0, x1);
                        const float p0 = e < lim ? ex2_approx(x0) : 0.f;
                        const float p1 = e + 1 < lim ? ex2_approx(x1) : 0.f;
                        acc[(i >> 1) & 3] = f2_add(acc[(i >> 1) & 3], f2_pack(p0, p1));
                        pk[cc * 16 + (i >> 1)] = pack2<KIND == kKindBF16>(p0, p1);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        pk[cc * 16 + i] = 0u;
                }
            }
            tmem_st32(tP + half * 32, pk);
        }
        float a0, a1, b0, b1;
        f2_unpack(f2_add(acc[0], acc[1]), a0, a1);
        f2_unpack(f2_add(acc[2], acc[3]), b0, b1);
        return (a0 + a1) + (b0 + b1);
    }
}

// KIND: element kind of Q, K, V and O (kKindF16, kKindBF16, or kKindTF32 for fp32 inputs and
// output); P has the kind of the inputs (one MMA takes A and B of one type).
template <int D, bool SPLIT, int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_tcgen05_kernel(const TcArgs args, const __grid_constant__ CUtensorMap tm_q,
                            const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v,
                            const __grid_constant__ SchedTable sched)
{
    constexpr bool TF32 = KIND == kKindTF32;
    constexpr int kES = elem_bytes<KIND>();
    using C = Cfg<D, kES>;
    using BB = Bars<D, kES>;
    // S = Q K^T: both K-major; O += P V: P from TMEM, V MN-major. A and B share one type.
    constexpr uint32_t kIdescS = TF32 ? idesc_tf32_f32(kBM, kBN, 0, 0)
                                      : idesc_f16_f32(kBM, kBN, 0, 0, KIND == kKindBF16);
    // (tf32: V is first transposed to K-major V^T, tf32 operands cannot be MN-major)
    constexpr uint32_t kIdescPV = TF32 ? idesc_tf32_f32(kBM, D, 0, 0)
                                       : idesc_f16_f32(kBM, D, 0, 1, KIND == kKindBF16);
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    unsigned char *smem = smem_raw + (base - raw_addr);
    const uint32_t sQ = base + C::kOffQ;
    const uint32_t sKV = base + C::kOffKV;
    const uint32_t sVT = base + C::kOffVT;
    const uint32_t sBar = base + C::kOffBar;
    auto bar = [&](int i) -> uint32_t { return sBar + 8u * static_cast<uint32_t>(i); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffBar + 8 * BB::kCount);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const uint32_t sClcResp = sBar + BB::kClcResp;
    Unit *unit_ring = reinterpret_cast<Unit *>(smem + C::kOffBar + BB::kUnitRing);
    // warps that take units from the ring: the MMA warp, the softmax warps, the transposers
    constexpr int kRingReaders = 1 + 8 + (TF32 ? 2 : 0);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const FwdParams &p = args.p;
    const uint64_t kWaitLimitNs = p.wait_limit_ns;

    if (warp == kProducerWarp && lane == 0) {
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kQStages; ++s) {
            mbar_init(bar(BB::kQFull + s), 1);
            mbar_init(bar(BB::kQEmpty + s), 1);
        }
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bar(BB::kKVFull + s), 1);
            mbar_init(bar(BB::kKVEmpty + s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(BB::kSFull + t), 1);
            mbar_init(bar(BB::kPFull + t), kBM);
            mbar_init(bar(BB::kSFree + t), kBM);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(bar(BB::kOReady + i), 1);
            mbar_init(bar(BB::kOEmpty + i), kBM);
        }
        mbar_init(bar(BB::kMmaDone), 1);
        for (int i = 0; i < kUnitSlots; ++i) {
            mbar_init(bar(BB::kUnitFull + i), 1);
            mbar_init(bar(BB::kUnitEmpty + i), kRingReaders);
        }
        mbar_init(bar(BB::kClc), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(BB::kVReady + i), 1);
            mbar_init(bar(BB::kVTFull + i), 64); // the 64 threads of the transposer warps
            mbar_init(bar(BB::kVTEmpty + i), 1);
        }
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    // Programmatic dependent launch: the setup above overlaps the end of the previous
    // kernel of the stream; no global memory is touched before griddep_wait.
    griddep_launch_dependents();
    griddep_wait();
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
    // The next unit of this CTA, for the roles other than the producer (whole warps). Static
    // schedule: from the table. Dynamic: from the producer's ring, in order; a unit with
    // n_kv < 0 marks the end.
    auto take = [&](UnitStream &st, Unit &U) -> bool {
        if (!args.dynamic)
            return stream_take(st, args, sched, U);
        if (!st.has)
            return false;
        const uint32_t slot = st.k % kUnitSlots;
        if (!warp_wait(bar(BB::kUnitFull + slot), (st.k / kUnitSlots) & 1u)) {
            st.has = false;
            return false;
        }
        U = unit_ring[slot];
        __syncwarp();
        if (lane == 0)
            mbar_arrive(bar(BB::kUnitEmpty + slot));
        ++st.k;
        if (U.n_kv < 0) {
            st.has = false;
            return false;
        }
        return true;
    };

    // The producer and MMA roles run on whole warps (converged control flow, warp-uniform
    // operands); one elected lane issues each TMA copy, tcgen05.mma and commit.
    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ TMA producer
        setmaxnreg_dec<RegSplit<D>::kControl>();
        uint32_t q_it = 0, kv_it = 0;
        bool ok = true;
        UnitStream us;
        stream_init(us, args, sched);
        Unit U;
        // Dynamic schedule: the producer decodes every unit of the CTA once and hands it to the
        // other roles through the ring. Its first unit is the CTA's own; each later one is the
        // unit of a CTA whose launch a cluster launch control request cancelled. One request
        // is in flight at a time, made as a unit is published and answered by the time that
        // unit's loads are issued; after an answer that cancelled nothing none is made.
        uint32_t pub = 0;           // units published
        uint32_t clc_par = 0;       // phase parity of the next answer
        bool clc_pending = false;   // a request is in flight
        int next_cta = blockIdx.x;  // the CTA whose unit comes next (-1: none)
        auto publish = [&](const Unit &X) -> bool {
            const uint32_t slot = pub % kUnitSlots;
            if (!warp_wait(bar(BB::kUnitEmpty + slot), ((pub / kUnitSlots) & 1u) ^ 1u))
                return false;
            if (lane == 0) {
                unit_ring[slot] = X;
                mbar_arrive(bar(BB::kUnitFull + slot)); // releases the unit's write
            }
            __syncwarp();
            ++pub;
            return true;
        };
        auto next = [&](Unit &X) -> bool {
            if (!args.dynamic)
                return stream_take(us, args, sched, X);
            if (next_cta < 0)
                return false;
            // (the CTA ids map to units through the host's order when it built one)
            X = decode_unit(args, sched.use ? static_cast<int>(sched.unit[next_cta]) : next_cta);
            if (!publish(X)) {
                ok = false;
                return false;
            }
            if (elect_one()) {
                // the last answer was read (generic proxy) before the request rewrites it
                asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
                mbar_arrive_expect_tx(bar(BB::kClc), 16);
                clc_try_cancel(sClcResp, bar(BB::kClc));
            }
            __syncwarp();
            clc_pending = true;
            return true;
        };
        auto answer = [&]() -> bool {
            if (!warp_wait(bar(BB::kClc), clc_par))
                return false;
            clc_par ^= 1u;
            clc_pending = false;
            const uint64_t *r = reinterpret_cast<const uint64_t *>(smem + C::kOffBar + BB::kClcResp);
            next_cta = clc_cancelled_x(r[0], r[1]);
            return true;
        };
        while (ok && next(U)) {
            if (args.dynamic && U.n_kv == 0) {
                if (!answer())
                    ok = false;
                continue;
            }
            if (U.n_kv == 0)
                continue;
            const uint32_t qs = q_it % C::kQStages;
            if (!warp_wait(bar(BB::kQEmpty + qs), ((q_it / C::kQStages) & 1u) ^ 1u)) {
                ok = false;
                break;
            }
            ++q_it;
            if (elect_one()) {
                mbar_arrive_expect_tx(bar(BB::kQFull + qs), 2 * C::kTileBytes);
#pragma unroll
                for (int t = 0; t < 2; ++t)
#pragma unroll
                    for (int bx = 0; bx < D / C::kBoxCols; ++bx)
                        tma_load_3d(sQ + (qs * 2 + t) * C::kTileBytes + bx * C::kBoxBytes, &tm_q,
                                    bar(BB::kQFull + qs), bx * C::kBoxCols, U.q0 + t * kBM, U.bh);
            }
            __syncwarp();
            for (int j = 0; j < U.n_kv && ok; ++j) {
#pragma unroll
                for (int kv = 0; kv < 2; ++kv) {
                    const uint32_t slot = kv_it % C::kStages;
                    const uint32_t ph = (kv_it / C::kStages) & 1u;
                    if (!warp_wait(bar(BB::kKVEmpty + slot), ph ^ 1u)) {
                        ok = false;
                        break;
                    }
                    if (elect_one()) {
                        mbar_arrive_expect_tx(bar(BB::kKVFull + slot), C::kTileBytes);
#pragma unroll
                        for (int bx = 0; bx < D / C::kBoxCols; ++bx)
                            tma_load_3d(sKV + slot * C::kTileBytes + bx * C::kBoxBytes,
                                        kv == 0 ? &tm_k : &tm_v, bar(BB::kKVFull + slot),
                                        bx * C::kBoxCols, (U.j0 + j) * kBN, U.kvh);
                    }
                    __syncwarp();
                    ++kv_it;
                }
            }
            if (args.dynamic && ok && !answer())
                ok = false;
        }
        if (args.dynamic) {
            if (ok) {
                Unit E = {};
                E.n_kv = -1; // the end of the CTA's units
                publish(E);
            }
            // (after an abort) the answer in flight lands before the CTA may leave
            if (clc_pending && lane == 0)
                mbar_wait(bar(BB::kClc), clc_par, nullptr, kWaitLimitNs);
            __syncwarp();
        }
        // Loads still in flight land before the CTA may leave (after an abort): wait,
        // bounded by time only, for the latest phase of every slot that was filled.
        if (lane == 0) {
            for (uint32_t i = q_it > C::kQStages ? q_it - C::kQStages : 0; i < q_it; ++i)
                mbar_wait(bar(BB::kQFull + i % C::kQStages), (i / C::kQStages) & 1u, nullptr, kWaitLimitNs);
            for (uint32_t i = kv_it > C::kStages ? kv_it - C::kStages : 0; i < kv_it; ++i)
                mbar_wait(bar(BB::kKVFull + i % C::kStages), (i / C::kStages) & 1u, nullptr, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        setmaxnreg_dec<RegSplit<D>::kControl>();
        uint32_t q_it = 0, kv_it = 0;
        uint32_t vt_it = 0; // V tiles consumed (tf32: V^T buffer vt_it & 1)
        // Phase parities kept as bit masks (no runtime-indexed local arrays):
        uint32_t p_par = 0;  // bit t: parity of the P-ready waits of tile t
        uint32_t oe_par = 0; // bit t*2+b: parity of the uses of O buffer b of tile t
        uint32_t u_par = 0;  // bit t: parity of the units tile t took part in
        uint32_t ob = 0;     // bit t: O buffer of tile t in the current unit
        bool ok = true;
        auto wait = [&](uint32_t b, uint32_t parity) {
            if (ok && !warp_wait(b, parity))
                ok = false;
            return ok;
        };
        uint32_t q_slot = 0;
        // Shared-memory descriptors, built once: the high word (stride byte offset,
        // version, swizzle layout) is the same for every operand; the low word is
        // (start address >> 4) | (leading byte offset >> 4) << 16, so stepping through
        // a tile is one add per instruction. Addresses stay below 2^18, so the start
        // field never carries into the leading-offset field.
        constexpr uint32_t kDescHi = ((8 * C::kRowBytes) >> 4) | (1u << 14) | (C::kSwizzle << 29);
        constexpr uint32_t kLboK = (16u >> 4) << 16;                            // K-major: unused
        constexpr uint32_t kLboV = (static_cast<uint32_t>(C::kBoxBytes) >> 4) << 16; // next 64 columns of d
        auto desc = [](uint32_t lo) -> uint64_t {
            return (static_cast<uint64_t>(kDescHi) << 32) | lo;
        };
        // S_t = Q_t K^T: K-major operands, 32 bytes (16 fp16 / 8 fp32 elements) per k-step
        // inside a swizzle row, a new box every kBoxCols / kKStep steps. (Issued by the
        // elected lane.)
        auto issue_s = [&](int t, uint32_t k_slot) {
            const uint32_t qlo = ((sQ + (q_slot * 2 + t) * C::kTileBytes) >> 4) | kLboK;
            const uint32_t klo = ((sKV + k_slot * C::kTileBytes) >> 4) | kLboK;
            const uint32_t d_tmem = tmem + (t ? C::kTmemS1 : C::kTmemS0);
            constexpr int kStepsPerBox = C::kBoxCols / C::kKStep;
#pragma unroll
            for (int kk = 0; kk < D / C::kKStep; ++kk) {
                constexpr int kBox16 = C::kBoxBytes >> 4;
                const uint32_t off = (kk / kStepsPerBox) * kBox16 + (kk % kStepsPerBox) * 2;
                if constexpr (TF32)
                    mma_ss_tf32(d_tmem, desc(qlo + off), desc(klo + off), kIdescS, kk > 0 ? 1u : 0u);
                else
                    mma_ss(d_tmem, desc(qlo + off), desc(klo + off), kIdescS, kk > 0 ? 1u : 0u);
            }
            mma_commit(bar(BB::kSFull + t));
        };
        // O_t += P_t V: P from TMEM (8 columns per k-step: 16 packed 16-bit keys, or 8 fp32
        // keys). 16-bit: V is MN-major, kKStep keys (rows) per k-step. tf32: V^T (buffer vt) is
        // K-major in four 32-key blocks of 4 KB, 8 keys (32 bytes) per k-step. (Issued by the
        // elected lane.)
        auto issue_pv = [&](int t, uint32_t v_slot, uint32_t vt, bool accumulate) {
            const uint32_t a_tmem = C::kSepP ? tmem + (t ? C::kTmemP1 : C::kTmemP0)
                                             : tmem + (t ? C::kTmemS1 : C::kTmemS0);
            const int b = static_cast<int>((ob >> t) & 1u);
            const uint32_t d_tmem = tmem + C::tmem_o(t, b);
            if constexpr (TF32) {
                const uint32_t vtlo = ((sVT + vt * C::kTileBytes) >> 4) | kLboK;
                constexpr uint32_t kBlock16 = (32u * D * 4u) >> 4; // one 32-key block of V^T
#pragma unroll
                for (int kk = 0; kk < kBN / C::kKStep; ++kk)
                    mma_ts_tf32(d_tmem, a_tmem + kk * 8, desc(vtlo + (kk / 4) * kBlock16 + (kk % 4) * 2),
                                kIdescPV, (accumulate || kk > 0) ? 1u : 0u);
            } else {
                const uint32_t vlo = ((sKV + v_slot * C::kTileBytes) >> 4) | kLboV;
#pragma unroll
                for (int kk = 0; kk < kBN / C::kKStep; ++kk)
                    mma_ts(d_tmem, a_tmem + kk * 8, desc(vlo + kk * ((C::kKStep * C::kRowBytes) >> 4)),
                           kIdescPV, (accumulate || kk > 0) ? 1u : 0u);
            }
            mma_commit(bar(BB::kOReady + t * 2 + b));
        };
        UnitStream us;
        stream_init(us, args, sched);
        // The next unit that has work (units without an allowed key need no MMA).
        auto take_work = [&](Unit &X) -> bool {
            while (take(us, X))
                if (X.n_kv > 0)
                    return true;
            return false;
        };
        // A unit's first S products: its Q buffer (q_slot is set to it) and first K tile,
        // then S_t(0) for every active tile.
        auto start_unit = [&](const Unit &X) -> bool {
            q_slot = q_it % C::kQStages;
            if (!wait(bar(BB::kQFull + q_slot), (q_it / C::kQStages) & 1u))
                return false;
            ++q_it;
            const uint32_t ks = kv_it % C::kStages;
            if (!wait(bar(BB::kKVFull + ks), (kv_it / C::kStages) & 1u))
                return false;
            ++kv_it;
            tc_fence_after();
            if (elect_one()) {
                for (int t = 0; t < 2; ++t)
                    if (kv_tiles(X, t) > 0)
                        issue_s(t, ks);
                mma_commit(bar(BB::kKVEmpty + ks));
                if (X.n_kv == 1)
                    mma_commit(bar(BB::kQEmpty + q_slot));
            }
            __syncwarp();
            return true;
        };
        Unit U, Un;
        bool have = take_work(U);
        if (have && !start_unit(U))
            have = false;
        if constexpr (C::kSepP) {
            // step j: S_t(j+1) = Q_t K_{j+1}^T for every tile as soon as its softmax has read
            // S_t(j) (SFree), then O_t += P_t(j) V_j once P_t(j) is out. The ring holds K_j, V_j,
            // K_{j+1}, ... in that order; K_{j+1} is taken before V_j.
            uint32_t sf_par = 0; // bit t: parity of the SFree waits of tile t
            while (ok && have) {
                const uint32_t uq_slot = q_slot;
                bool have_next = false;
                for (int j = 0; j < U.n_kv && ok; ++j) {
                    const uint32_t v_pos = kv_it;
                    const uint32_t v_slot = v_pos % C::kStages;
                    const bool has_next = j + 1 < U.n_kv;
                    const uint32_t k_slot = (v_pos + 1) % C::kStages;
                    if (has_next) {
                        bool k_ready = false;
                        for (int t = 0; t < 2 && ok; ++t) {
                            if (j + 1 >= kv_tiles(U, t))
                                continue;
                            if (!wait(bar(BB::kSFree + t), (sf_par >> t) & 1u))
                                break;
                            sf_par ^= 1u << t;
                            if (!k_ready) {
                                if (!wait(bar(BB::kKVFull + k_slot), ((v_pos + 1) / C::kStages) & 1u))
                                    break;
                                k_ready = true;
                            }
                            tc_fence_after();
                            if (elect_one())
                                issue_s(t, k_slot);
                            __syncwarp();
                        }
                        if (!ok)
                            break;
                    }
                    if (!wait(bar(BB::kKVFull + v_slot), (v_pos / C::kStages) & 1u))
                        break;
                    kv_it = v_pos + (has_next ? 2u : 1u);
                    for (int t = 0; t < 2 && ok; ++t) {
                        if (j >= kv_tiles(U, t))
                            continue;
                        if (j == 0) {
                            // the epilogue of the unit that last used this tile's O is done
                            const int ob_i = t * 2;
                            if (!wait(bar(BB::kOEmpty + ob_i), ((oe_par >> ob_i) & 1u) ^ 1u))
                                break;
                            oe_par ^= 1u << ob_i;
                        }
                        if (!wait(bar(BB::kPFull + t), (p_par >> t) & 1u))
                            break;
                        p_par ^= 1u << t;
                        tc_fence_after();
                        if (elect_one())
                            issue_pv(t, v_slot, 0u, j > 0);
                        __syncwarp();
                    }
                    if (!ok)
                        break;
                    if (elect_one()) {
                        mma_commit(bar(BB::kKVEmpty + v_slot));
                        if (has_next) {
                            mma_commit(bar(BB::kKVEmpty + k_slot));
                            if (j + 2 == U.n_kv)
                                mma_commit(bar(BB::kQEmpty + uq_slot));
                        }
                    }
                    __syncwarp();
                    if (!has_next) {
                        // The next unit is taken only now (the dynamic schedule's producer
                        // publishes it once this unit's loads are all issued).
                        have_next = take_work(Un);
                        if (have_next && !start_unit(Un))
                            break;
                    }
                }
                U = Un;
                have = have_next;
            }
            have = false;
        }
        while (ok && have) {
            const uint32_t uq_slot = q_slot; // this unit's Q buffer
            ob = C::kOBufs == 2 ? u_par : 0u;
            bool have_next = false;
            // step j: O_t += P_t(j) V_j, then S_t(j+1) = Q_t K_{j+1}^T; a tile whose
            // causal range ends earlier drops out of the later steps. After the last
            // step the next unit's first S products follow at once, so the softmax
            // warps never wait at a unit boundary for the MMA warp's bookkeeping.
            for (int j = 0; j < U.n_kv && ok; ++j) {
                const uint32_t v_slot = kv_it % C::kStages;
                if (!wait(bar(BB::kKVFull + v_slot), (kv_it / C::kStages) & 1u))
                    break;
                ++kv_it;
                const uint32_t vt = vt_it & 1u; // tf32: the V^T buffer of this V tile
                if constexpr (TF32) {
                    // hand V_j to the transposer warps (in order, so their waits never alias)
                    if (elect_one())
                        mbar_arrive(bar(BB::kVReady + vt));
                    __syncwarp();
                }
                bool vt_ready = false;
                const bool has_next = j + 1 < U.n_kv;
                bool k_ready = false;
                uint32_t k_slot = 0;
                for (int t = 0; t < 2 && ok; ++t) {
                    if (j >= kv_tiles(U, t))
                        continue;
                    if (j == 0) {
                        // the epilogue of the last unit that used this O buffer is done
                        const int ob_i = t * 2 + static_cast<int>((ob >> t) & 1u);
                        if (!wait(bar(BB::kOEmpty + ob_i), ((oe_par >> ob_i) & 1u) ^ 1u))
                            break;
                        oe_par ^= 1u << ob_i;
                    }
                    if (!wait(bar(BB::kPFull + t), (p_par >> t) & 1u))
                        break;
                    p_par ^= 1u << t;
                    if constexpr (TF32) {
                        if (!vt_ready) {
                            if (!wait(bar(BB::kVTFull + vt), (vt_it >> 1) & 1u))
                                break;
                            vt_ready = true;
                        }
                    }
                    tc_fence_after();
                    if (elect_one())
                        issue_pv(t, v_slot, vt, j > 0);
                    __syncwarp();
                    if (j + 1 < kv_tiles(U, t)) {
                        if (!k_ready) {
                            k_slot = kv_it % C::kStages;
                            if (!wait(bar(BB::kKVFull + k_slot), (kv_it / C::kStages) & 1u))
                                break;
                            ++kv_it;
                            k_ready = true;
                            tc_fence_after();
                        }
                        if (elect_one())
                            issue_s(t, k_slot);
                        __syncwarp();
                    }
                }
                if (!ok)
                    break;
                if (elect_one()) {
                    mma_commit(bar(BB::kKVEmpty + v_slot));
                    if constexpr (TF32)
                        mma_commit(bar(BB::kVTEmpty + vt));
                    if (has_next) {
                        // the tile with the most K/V tiles always consumed K_{j+1} above
                        mma_commit(bar(BB::kKVEmpty + k_slot));
                        if (j + 2 == U.n_kv)
                            mma_commit(bar(BB::kQEmpty + uq_slot));
                    }
                }
                __syncwarp();
                ++vt_it;
                if (!has_next) {
                    // The next unit is taken only now (the dynamic schedule's producer
                    // publishes it once this unit's loads are all issued).
                    have_next = take_work(Un);
                    if (have_next && !start_unit(Un))
                        break;
                }
            }
            for (int t = 0; t < 2; ++t)
                if (kv_tiles(U, t) > 0)
                    u_par ^= 1u << t;
            U = Un;
            have = have_next;
        }
        // Every MMA this warp issued is complete before TMEM is released (bounded by
        // time only: this wait must not give up early on an abort).
        if (elect_one())
            mma_commit(bar(BB::kMmaDone));
        __syncwarp();
        mbar_wait(bar(BB::kMmaDone), 0, nullptr, kWaitLimitNs);
        __syncwarp();
    } else if (warp >= 8) {
        setmaxnreg_dec<RegSplit<D>::kControl>(); // warps 10 and 11 of the control warpgroup
        if constexpr (TF32) {
            // ------------------------------------------------------------ V transposer (tf32)
            // V_j [128 keys x D] (TMA layout: 128-byte rows, 128-byte swizzle) -> V^T [D x 128
            // keys], K-major: four 32-key blocks of D rows x 128 bytes, same swizzle. Each
            // thread moves four 4 x 4 blocks (four 16-byte loads, a register transpose, four
            // 16-byte stores). V_j's stage is known in order from the MMA warp (VReady), so
            // no wait here can mistake an old phase for a new one.
            static_assert(D == 32, "the tf32 path is built for d = 32");
            const int tt = static_cast<int>(threadIdx.x) - 10 * 32; // 0..63
            uint32_t g = 0; // V tiles transposed
            bool ok = true;
            UnitStream us;
            stream_init(us, args, sched);
            Unit U;
            while (ok && take(us, U)) {
                for (int j = 0; j < U.n_kv; ++j) {
                    const uint32_t vt = g & 1u, use = g >> 1;
                    if (!warp_wait(bar(BB::kVReady + vt), use & 1u) ||
                        !warp_wait(bar(BB::kVTEmpty + vt), (use & 1u) ^ 1u)) {
                        ok = false;
                        break;
                    }
                    const uint32_t kv = 2 * g + 1; // K and V tiles alternate in the ring
                    const unsigned char *src = smem + C::kOffKV + (kv % C::kStages) * C::kTileBytes;
                    unsigned char *dst = smem + C::kOffVT + vt * C::kTileBytes;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int blk = tt + 64 * i;
                        const int rb = blk >> 3, cb = blk & 7; // keys 4rb.., dims 4cb..
                        float4 x[4];
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const int key = 4 * rb + r;
                            x[r] = *reinterpret_cast<const float4 *>(src + key * 128 + ((cb ^ (key & 7)) << 4));
                        }
                        const float4 y[4] = {make_float4(x[0].x, x[1].x, x[2].x, x[3].x),
                                             make_float4(x[0].y, x[1].y, x[2].y, x[3].y),
                                             make_float4(x[0].z, x[1].z, x[2].z, x[3].z),
                                             make_float4(x[0].w, x[1].w, x[2].w, x[3].w)};
#pragma unroll
                        for (int n = 0; n < 4; ++n) {
                            const int dim = 4 * cb + n;
                            *reinterpret_cast<float4 *>(dst + (rb >> 3) * (32 * D * 4) + dim * 128 +
                                                        (((rb & 7) ^ (dim & 7)) << 4)) = y[n];
                        }
                    }
                    // the writes are read by tcgen05.mma (async proxy)
                    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
                    mbar_arrive(bar(BB::kVTFull + vt));
                    ++g;
                }
            }
        }
    } else {
        // ------------------------------------------------------------ softmax warpgroups
        setmaxnreg_inc<RegSplit<D>::kSoftmax>();
        const int t = warp >> 2;         // Q tile of this warpgroup
        const int wq = warp & 3;         // TMEM lane quarter
        const int rt = wq * 32 + lane;   // row within the Q tile = TMEM lane
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const uint32_t tS = lane_base + (t ? C::kTmemS1 : C::kTmemS0);
        // where P_t goes: its own columns (separate P) or over the first half of S_t
        const uint32_t tP = C::kSepP ? lane_base + (t ? C::kTmemP1 : C::kTmemP0) : tS;
        const float scale = p.scale_log2;
        const int diag = p.Nk - p.N; // causal: query i sees keys j <= i + diag
        // packed query groups: row r is query r % qrows, whose diagonal is at Nk - qrows; every
        // tile holds a query 0, the row that sees the fewest keys
        const int qdiag = p.qrows ? p.Nk - p.qrows : diag;
        uint32_t s_it = 0;
        uint32_t pv_par = 0; // bit b: parity of the PV products committed into O buffer b
        uint32_t ucnt = 0;   // units in which this tile took part
        bool ok = true;
        // tcgen05.ld/st are warp-collective (.sync.aligned): every branch around them, and
        // every decision to give up, is made uniform across the warp first.
        auto wait_all = [&](uint32_t b, uint32_t parity) -> bool {
            bool r = mbar_wait(b, parity, abort_flag, kWaitLimitNs);
            r = __all_sync(0xffffffffu, r);
            if (!r)
                fail();
            return r;
        };
        // A unit whose last P has been released but whose epilogue has not run yet. With two
        // O buffers the epilogue is deferred until the next unit's first P is out, so that
        // waiting for the last PV product and reading O overlap with the next unit's first
        // softmax step.
        struct Pending {
            bool valid;
            int bh, row, b, split;
            uint32_t last_par; // phase parity of its last PV product in buffer b
            float l, m_ref;
        } pend;
        pend.valid = false;
        auto finish = [&](const Pending &pe) -> bool {
            if (!wait_all(bar(BB::kOReady + t * 2 + pe.b), pe.last_par))
                return false;
            tc_fence_after();
            const uint32_t tO = lane_base + C::tmem_o(t, pe.b);
            const float inv = pe.l > 0.f ? 1.f / pe.l : 0.f;
            // Each thread writes its own row, so a warp's store touches 32 rows: 32-byte stores
            // (when the output is 32-byte aligned; rows are multiples of 32 bytes) fill whole
            // sectors and take half the sector requests of 16-byte ones.
            auto store_f32 = [&](float *dst, const uint32_t (&ov)[32], bool v8) {
                if (v8) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8)
                        st_global_v8(dst + e, __float_as_uint(__uint_as_float(ov[e]) * inv),
                                     __float_as_uint(__uint_as_float(ov[e + 1]) * inv),
                                     __float_as_uint(__uint_as_float(ov[e + 2]) * inv),
                                     __float_as_uint(__uint_as_float(ov[e + 3]) * inv),
                                     __float_as_uint(__uint_as_float(ov[e + 4]) * inv),
                                     __float_as_uint(__uint_as_float(ov[e + 5]) * inv),
                                     __float_as_uint(__uint_as_float(ov[e + 6]) * inv),
                                     __float_as_uint(__uint_as_float(ov[e + 7]) * inv));
                } else {
                    float4 *d4 = reinterpret_cast<float4 *>(dst);
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        d4[e >> 2] = make_float4(__uint_as_float(ov[e]) * inv, __uint_as_float(ov[e + 1]) * inv,
                                                 __uint_as_float(ov[e + 2]) * inv, __uint_as_float(ov[e + 3]) * inv);
                }
            };
            if constexpr (SPLIT) {
                // The range's O / l in fp32 and its logsumexp, for the merge.
                const size_t r = static_cast<size_t>(pe.split) * args.p.B * args.p.H * p.N +
                                 static_cast<size_t>(pe.bh) * p.N + pe.row;
                float *orow = args.opart + r * D;
                const bool v8 = (reinterpret_cast<uintptr_t>(args.opart) & 31u) == 0;
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t ov[32];
                    tmem_ld32(tO + c0, ov);
                    if (pe.row < p.N)
                        store_f32(orow + c0, ov, v8);
                }
                tc_fence_before();
                mbar_arrive(bar(BB::kOEmpty + t * 2 + pe.b));
                if (pe.row < p.N)
                    args.lpart[r] = pe.l > 0.f ? (pe.m_ref + log2f(pe.l)) * kLn2 : -INFINITY;
                return true;
            }
            if constexpr (TF32) {
                // fp32 output: O / l as it is
                float *orow = reinterpret_cast<float *>(p.o) + (static_cast<size_t>(pe.bh) * p.N + pe.row) * D;
                const bool v8 = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t ov[32];
                    tmem_ld32(tO + c0, ov);
                    if (pe.row < p.N)
                        store_f32(orow + c0, ov, v8);
                }
                tc_fence_before();
                mbar_arrive(bar(BB::kOEmpty + t * 2 + pe.b));
                if (p.lse && pe.row < p.N)
                    p.lse[static_cast<size_t>(pe.bh) * p.N + pe.row] =
                        pe.l > 0.f ? (pe.m_ref + log2f(pe.l)) * kLn2 : -INFINITY;
                return true;
            }
            __half *orow = p.o + (static_cast<size_t>(pe.bh) * p.N + pe.row) * D;
            const bool v8 = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;
            constexpr int kChunk = D < 64 ? D : 64; // O columns per TMEM load
#pragma unroll
            for (int half = 0; half < D / kChunk; ++half) {
                uint32_t ov[kChunk];
                if constexpr (kChunk == 64)
                    tmem_ld64(tO + half * 64, ov);
                else
                    tmem_ld32(tO, ov);
                uint32_t h[kChunk / 2];
#pragma unroll
                for (int e = 0; e < kChunk; e += 2)
                    h[e >> 1] = pack2<KIND == kKindBF16>(__uint_as_float(ov[e]) * inv, __uint_as_float(ov[e + 1]) * inv);
                if (pe.row < p.N) {
                    if (v8) {
#pragma unroll
                        for (int c = 0; c < kChunk / 16; ++c)
                            st_global_v8(orow + half * kChunk + c * 16, h[8 * c], h[8 * c + 1], h[8 * c + 2],
                                         h[8 * c + 3], h[8 * c + 4], h[8 * c + 5], h[8 * c + 6], h[8 * c + 7]);
                    } else {
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + half * kChunk);
#pragma unroll
                        for (int c = 0; c < kChunk / 8; ++c)
                            dst[c] = make_uint4(h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(bar(BB::kOEmpty + t * 2 + pe.b));
            if (p.lse && pe.row < p.N)
                p.lse[static_cast<size_t>(pe.bh) * p.N + pe.row] =
                    pe.l > 0.f ? (pe.m_ref + log2f(pe.l)) * kLn2 : -INFINITY;
            return true;
        };
        UnitStream us;
        stream_init(us, args, sched);
        Unit U;
        while (ok && take(us, U)) {
            const int n_kv = kv_tiles(U, t);
            if (n_kv == 0) {
                // Nothing to accumulate: rows with no allowed key get O = 0 and lse = -inf
                // (rows past N, of a tile that lies beyond the sequence, are not written).
                const int row = U.q0 + t * kBM + rt;
                if (SPLIT && row < p.N) {
                    // no key of this range for the tile: weight 0 in the merge
                    const size_t r = static_cast<size_t>(U.split) * args.p.B * args.p.H * p.N +
                                     static_cast<size_t>(U.bh) * p.N + row;
                    float4 *orow = reinterpret_cast<float4 *>(args.opart + r * D);
#pragma unroll
                    for (int c = 0; c < D / 4; ++c)
                        orow[c] = make_float4(0.f, 0.f, 0.f, 0.f);
                    args.lpart[r] = -INFINITY;
                } else if (row < p.N) {
                    // D elements of kES bytes: D * kES / 16 vectors of 16 bytes
                    uint4 z = make_uint4(0, 0, 0, 0);
                    uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<char *>(p.o) +
                                                           (static_cast<size_t>(U.bh) * p.N + row) * D * kES);
#pragma unroll
                    for (int c = 0; c < D * kES / 16; ++c)
                        dst[c] = z;
                    if (p.lse)
                        p.lse[static_cast<size_t>(U.bh) * p.N + row] = -INFINITY;
                }
                continue;
            }
            const int b = C::kOBufs == 2 ? static_cast<int>(ucnt & 1u) : 0;
            const uint32_t tO = lane_base + C::tmem_o(t, b);
            const int row = U.q0 + t * kBM + rt;
            const int tile_row0 = U.q0 + t * kBM;
            // causal: this row's last allowed key, and the key past which some row of the tile
            // needs the element mask (fixed for the unit)
            const int row_diag = (p.qrows ? row % p.qrows : row) + qdiag;
            const int mask_from = p.qrows ? qdiag : tile_row0 + diag;
            float m_ref = -INFINITY; // reference max of the exponentials (log2 units)
            float l = 0.f;
            for (int j = 0; j < n_kv; ++j) {
                if (!wait_all(bar(BB::kSFull + t), s_it & 1u)) {
                    ok = false;
                    break;
                }
                ++s_it;
                tc_fence_after();
                const int kv0 = (U.j0 + j) * kBN;
                const bool need_mask = (kv0 + kBN > U.L) || (p.causal && kv0 + kBN - 1 > mask_from);
                int lim = U.L - kv0; // keys [kv0, kv0 + lim) are allowed for this row
                if (p.causal)
                    lim = min(lim, row_diag - kv0 + 1);

                uint32_t sv[kBN];
                tmem_ld128(tS, sv);
                if constexpr (C::kSepP) {
                    // S_t(j) is read: the MMA warp may compute S_t(j+1) over it now
                    if (j + 1 < n_kv) {
                        tc_fence_before();
                        mbar_arrive(bar(BB::kSFree + t));
                    }
                }
                const float mx = need_mask ? row_max(sv, scale, lim) : row_max_full(sv, scale);
                // Lazy correction: a row moves its reference only when its max grew by more
                // than 2^8 over it; O and l are rescaled together, so the result is exact.
                const bool want = mx > m_ref + kRescaleLog2;
                const float alpha = want ? ex2_approx(m_ref - mx) : 1.f;
                const float m_new = want ? mx : m_ref;
                const float neg_m = m_new == -INFINITY ? 0.f : -m_new;

                if constexpr (C::kSepP) {
                    // P_t(j) is written over P_t(j-1): the PV product reading it must be done
                    if (j > 0) {
                        if (!wait_all(bar(BB::kOReady + t * 2 + b), ((pv_par >> b) & 1u) ^ 1u)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                }
                // P = exp2(S * scale - m_ref) as fp16, written over the first 64 columns of S
                // (or into P_t's own columns)
                const float rs = need_mask ? exp_pack<KIND>(sv, scale, neg_m, lim, tP)
                                           : exp_pack_full<KIND>(sv, scale, neg_m, tP);
                // O holds the PV products of earlier tiles; rescale it (after the last of
                // them is done) before this tile's P is released to the MMA warp. The warp
                // does it together when any of its rows needs it (tcgen05.ld/st are
                // warp-collective).
                if (__any_sync(0xffffffffu, want && l > 0.f)) {
                    if (!wait_all(bar(BB::kOReady + t * 2 + b), ((pv_par >> b) & 1u) ^ 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t v[32];
                        tmem_ld32(tO + c * 32, v);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                        tmem_st32(tO + c * 32, v);
                    }
                }
                l = l * alpha + rs;
                m_ref = m_new;
                tmem_wait_st();
                tc_fence_before();
                // (self-test hook: withholding the first arrival makes the MMA warp's bounded
                // wait run out; never set in normal use)
                if (!(p.inject_missing_arrive && j == 0))
                    mbar_arrive(bar(BB::kPFull + t));
                pv_par ^= 1u << b;
                // the previous unit's epilogue, now that this unit's first P is out
                if (j == 0 && pend.valid) {
                    if (!finish(pend)) {
                        ok = false;
                        break;
                    }
                    pend.valid = false;
                }
            }
            if (!ok)
                break;
            Pending done;
            done.valid = true;
            done.bh = U.bh;
            done.row = row;
            done.b = b;
            done.split = U.split;
            done.last_par = ((pv_par >> b) & 1u) ^ 1u;
            done.l = l;
            done.m_ref = m_ref;
            ++ucnt;
            if (C::kOBufs == 1) {
                // One O buffer: the next unit's PV products wait for this epilogue, so it runs now.
                if (!finish(done))
                    break;
            } else {
                pend = done;
            }
        }
        if (ok && pend.valid)
            finish(pend);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp)
        tmem_dealloc(tmem, C::kTmemCols);
}

// [heads, rows, D] viewed as a 3-D tensor (D innermost): Q is [B*H, N, D], K and V
// [B*Hkv, Nk, D]; boxes of 128 rows x one swizzle row (128 bytes with a 128-byte swizzle, or
// 64 bytes with a 64-byte swizzle for fp16 at D = 32); rows past the end read as zero.
template <int D, int KIND>
bool encode_map(CUtensorMap *m, const void *ptr, int BH, int N)
{
    using C = Cfg<D, elem_bytes<KIND>()>;
    auto enc = tensor_map_encoder();
    if (!enc)
        return false;
    const CUtensorMapDataType dt = KIND == kKindTF32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : KIND == kKindBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    constexpr cuuint64_t kES = elem_bytes<KIND>();
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * kES,
                             static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(D) * kES};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(C::kBoxCols), static_cast<cuuint32_t>(kBM), 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void *>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE,
               C::kRowBytes < 128 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Heads per block of the unit order: keep the K/V of the heads in flight within about
// 16 MB of L2, so the query-tile pairs of one head reuse its K/V from L2. G consecutive
// query heads share one K/V head. (Measured on GB300, three alternating runs each, prefill in
// TFLOP/s: 48 MB 1259, 24 MB 1301, 16 MB 1311-1322, 12 MB 1289-1295; at 16 MB the bf16 prefill,
// grouped-query and chunked prefill are also the fastest of these.)
int head_block_for(int BH, int Nk, int D, int G)
{
    const long long kv_head = 4LL * Nk * D; // K and V of one key/value head, fp16
    const long long hblk = (16LL << 20) / (kv_head > 0 ? kv_head : 1) * G;
    return static_cast<int>(hblk < 1 ? 1 : (hblk > BH ? BH : hblk));
}

// Run (of G over T tiles laid end to end, run c covering [c T / G, (c + 1) T / G)) that holds
// tile t.
long long run_of(long long t, long long T, long long G) { return ((t + 1) * G - 1) / T; }

// K/V tiles per (batch*head, pair) as the host sees them (key lengths taken as Nk), when every
// pair has the same count (no causal mask, or a single pair); 0 otherwise.
int uniform_pair_tiles(int N, int Nk, int causal)
{
    const int n_pairs = (N + 2 * kBM - 1) / (2 * kBM);
    if (!causal)
        return (Nk + kBN - 1) / kBN;
    if (n_pairs != 1)
        return 0;
    const int e0 = std::max(0, std::min(Nk, kBM + Nk - N));
    const int e1 = std::max(0, std::min(Nk, 2 * kBM + Nk - N));
    const int f0 = (e0 + kBN - 1) / kBN;
    const int f1 = kBM < N ? (e1 + kBN - 1) / kBN : 0;
    return std::max(f0, f1);
}

// Longest run of K/V tiles (in tiles, plus a per-unit cost) a CTA gets: balanced runs of
// ceil(T / G) tiles, each starting ceil(run / nf) + 1 units at most, or equal ranges of a
// pair in waves.
// Cost of a unit start in K/V tiles, fitted on GB300 decode shapes (d = 128, 8192 keys, 32 query
// heads over 8): balanced runs were faster at 108 tiles per SM (188 vs 209 us) and slower at
// 27-47 (70 vs 67 us), which puts it between 5 and 20.
constexpr long long kUnitCostTiles = 8;
// Units per SM from which the dynamic schedule is used (measured: 256 units on 152 SMs ran 1 %
// slower dealt dynamically than by the static table; 1024 to 4096 units ran 1-4 % faster).
constexpr int kDynamicUnitsPerSm = 3;
long long balanced_makespan(long long pairs, int nf, int G)
{
    const long long T = pairs * nf;
    const long long run = (T + G - 1) / G;
    return run + ((run + nf - 1) / nf + 1) * kUnitCostTiles;
}
long long uniform_makespan(long long pairs, int nf, int sms, int S)
{
    const long long units = pairs * S;
    const long long waves = (units + sms - 1) / sms;
    return waves * ((nf + S - 1) / S + kUnitCostTiles);
}

// Most runs that touch one pair (the ranges per pair a balanced split needs).
int balanced_slots(long long pairs, int nf, int G)
{
    const long long T = pairs * nf;
    long long mx = 0;
    for (long long w = 0; w < pairs; ++w)
        mx = std::max(mx, run_of(w * nf + nf - 1, T, G) - run_of(w * nf, T, G) + 1);
    return static_cast<int>(mx);
}

} // namespace

// Balanced split-KV for a launch with n_splits ranges per pair: the per-pair K/V tile count
// when the balanced runs fit in n_splits ranges, fit the schedule table and finish sooner than
// n_splits equal ranges per pair; 0 for the equal ranges.
int splitkv_balanced_runs(int BH, int N, int Nk, int causal, int sms, int n_splits)
{
    const int nf = uniform_pair_tiles(N, Nk, causal);
    if (nf < 2 || n_splits < 2 || sms < 1)
        return 0;
    const long long pairs = static_cast<long long>(BH) * ((N + 2 * kBM - 1) / (2 * kBM));
    const long long T = pairs * nf;
    const int G = static_cast<int>(T < sms ? T : sms);
    if (G > kMaxCtas || pairs * n_splits > kMaxSchedUnits || pairs > 0xffff)
        return 0;
    if (balanced_slots(pairs, nf, G) > n_splits)
        return 0;
    return balanced_makespan(pairs, nf, G) < uniform_makespan(pairs, nf, sms, n_splits) ? nf : 0;
}

// Ranges per pair for the automatic split-KV choice when balanced runs beat every equal split
// (the slots they need), else 0.
int splitkv_balanced_auto(int BH, int N, int Nk, int causal, int sms, int max_splits)
{
    const int nf = uniform_pair_tiles(N, Nk, causal);
    if (nf < 2 || sms < 1)
        return 0;
    const long long pairs = static_cast<long long>(BH) * ((N + 2 * kBM - 1) / (2 * kBM));
    const long long T = pairs * nf;
    const int G = static_cast<int>(T < sms ? T : sms);
    const int slots = balanced_slots(pairs, nf, G);
    if (slots < 2 || slots > max_splits)
        return 0;
    long long best_uniform = uniform_makespan(pairs, nf, sms, 1);
    for (int S = 2; S <= max_splits && S <= nf; ++S)
        best_uniform = std::min(best_uniform, uniform_makespan(pairs, nf, sms, S));
    return splitkv_balanced_runs(BH, N, Nk, causal, sms, slots) > 0 &&
                   balanced_makespan(pairs, nf, G) < best_uniform
               ? slots
               : 0;
}

namespace {

// Weight of every unit in the device's unit order (head block by head block, heaviest pair first
// inside a block, the key ranges of a pair next to each other): its count of (Q tile, K/V tile)
// steps plus kUnitCostTiles, the measured cost of starting a unit; key lengths are not known on
// the host and are taken as Nk.
std::vector<long long> unit_weights(int BH, int N, int Nk, int causal, int head_block, int n_pairs, int S)
{
    const int n_units = BH * n_pairs * S;
    const int per_block = head_block * n_pairs * S;
    std::vector<long long> wts(n_units);
    for (int u = 0; u < n_units; ++u) {
        const int blk = u / per_block;
        const int ws = u - blk * per_block;
        const int split = ws % S;
        const int w = ws / S;
        const int hb = std::min(head_block, BH - blk * head_block);
        const int pair = n_pairs - 1 - w / hb;
        const int q0 = pair * 2 * kBM;
        int e0 = Nk, e1 = Nk;
        if (causal) {
            e0 = std::max(0, std::min(Nk, q0 + kBM + Nk - N));
            e1 = std::max(0, std::min(Nk, q0 + 2 * kBM + Nk - N));
        }
        const int f0 = (e0 + kBN - 1) / kBN;
        const int f1 = q0 + kBM < N ? (e1 + kBN - 1) / kBN : 0;
        const int nf = std::max(f0, f1);
        const int j0 = split * nf / S, j1 = (split + 1) * nf / S;
        wts[u] = std::max(0, std::min(j1, f0) - j0) + std::max(0, std::min(j1, f1) - j0) + kUnitCostTiles;
    }
    return wts;
}

// Largest-first assignment of the units to the least loaded CTA. The units are taken in
// the device's unit order (head block by head block, heaviest pair first inside a
// block, the key ranges of a pair next to each other), so every CTA works on the same head
// block at about the same time. The weight of a unit is its count of (Q tile, K/V tile)
// steps plus a fixed per-unit cost; key lengths are not known on the host and are taken as Nk.
void build_schedule(SchedTable &t, int BH, int N, int Nk, int causal, int head_block, int n_pairs,
                    int n_splits, int grid)
{
    const std::vector<long long> wts = unit_weights(BH, N, Nk, causal, head_block, n_pairs, n_splits);
    const int n_units = static_cast<int>(wts.size());
    using Slot = std::pair<long long, int>; // (load, cta)
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
    for (int c = 0; c < grid; ++c)
        heap.push({0, c});
    std::vector<std::vector<uint16_t>> lists(grid);
    for (int u = 0; u < n_units; ++u) {
        Slot sl = heap.top();
        heap.pop();
        lists[sl.second].push_back(static_cast<uint16_t>(u));
        heap.push({sl.first + wts[u], sl.second});
    }
    t.use = 1;
    int k = 0;
    for (int c = 0; c < grid; ++c) {
        t.off[c] = static_cast<uint16_t>(k);
        for (uint16_t u : lists[c])
            t.unit[k++] = u;
    }
    t.off[grid] = static_cast<uint16_t>(k);
}

// Balanced split-KV schedule (see TcArgs::bal_chunks): CTA c takes, in order, the part of
// every pair that run c touches; the ranges a pair has no run for are empty units (they
// write the zero-weight partials the merge expects), taken by the CTA of the pair's last run.
void build_balanced_schedule(SchedTable &t, long long pairs, int nf, int G, int S)
{
    const long long T = pairs * nf;
    std::vector<std::vector<uint16_t>> lists(G);
    for (int c = 0; c < G; ++c) {
        const long long lo = c * T / G, hi = (c + 1) * T / G;
        if (lo >= hi)
            continue;
        for (long long w = lo / nf; w <= (hi - 1) / nf; ++w)
            lists[c].push_back(static_cast<uint16_t>(w * S + (c - run_of(w * nf, T, G))));
    }
    for (long long w = 0; w < pairs; ++w) {
        const long long c0 = run_of(w * nf, T, G), c1 = run_of(w * nf + nf - 1, T, G);
        for (long long k = c1 - c0 + 1; k < S; ++k)
            lists[c1].push_back(static_cast<uint16_t>(w * S + k));
    }
    t.use = 1;
    int k = 0;
    for (int c = 0; c < G; ++c) {
        t.off[c] = static_cast<uint16_t>(k);
        for (uint16_t u : lists[c])
            t.unit[k++] = u;
    }
    t.off[G] = static_cast<uint16_t>(k);
}

// Order of the units for the dynamic schedule: CTA id c runs unit unit[c]. The units come in
// the device's unit order, except that the last ~20 % of the work, from a head-block boundary
// on and over at most three head blocks, is sorted heaviest first across its blocks. The
// scheduler hands out CTAs that have not started roughly in id order (measured: ascending,
// shuffled within ~100 ids), so the launch ends on the lightest units whatever the shuffle; in
// block order alone a heavy unit of the last block could start last. (A larger sorted share
// mixes more head blocks in L2: 50 % measured 1.4 % slower on prefill.)
void build_dynamic_order(SchedTable &t, int BH, int N, int Nk, int causal, int head_block, int n_pairs,
                         int n_splits)
{
    const std::vector<long long> wts = unit_weights(BH, N, Nk, causal, head_block, n_pairs, n_splits);
    const int n_units = static_cast<int>(wts.size());
    const int per_block = head_block * n_pairs * n_splits;
    long long total = 0;
    for (long long w : wts)
        total += w;
    int cut = 0;
    long long acc = 0;
    for (int u = n_units - 1; u >= 0; --u) {
        acc += wts[u];
        if (acc * 10 > total * 2) {
            cut = u + 1;
            break;
        }
    }
    cut = cut / per_block * per_block;
    // at most three head blocks (48 MB of K/V) are mixed, so the tail's K/V stays in L2 (six
    // one-head blocks of the N = 32768 workload, sorted together, read K/V 3x from DRAM)
    cut = std::max(cut, n_units - 3 * per_block);
    std::vector<int> order(n_units);
    for (int u = 0; u < n_units; ++u)
        order[u] = u;
    std::stable_sort(order.begin() + cut, order.end(), [&](int a, int b) { return wts[a] > wts[b]; });
    t.use = 1;
    for (int c = 0; c < n_units; ++c)
        t.unit[c] = static_cast<uint16_t>(order[c]);
}

// Schedules are cached per shape (they depend on B*H, N, Nk, the head block, causal, the
// split count, the SM count and the balanced run length only).
std::mutex g_sched_mutex;
std::map<std::tuple<int, int, int, int, int, int, int, int>, std::shared_ptr<SchedTable>> g_sched_cache;

std::shared_ptr<SchedTable> schedule_for(int BH, int N, int Nk, int causal, int head_block, int n_pairs,
                                         int n_splits, int grid, int bal_nfull = 0)
{
    auto key = std::make_tuple(BH, N, Nk, causal, head_block, n_splits, grid, bal_nfull);
    std::lock_guard<std::mutex> lock(g_sched_mutex);
    auto it = g_sched_cache.find(key);
    if (it != g_sched_cache.end())
        return it->second;
    auto t = std::make_shared<SchedTable>();
    memset(t.get(), 0, sizeof(SchedTable));
    const long long n_units = static_cast<long long>(BH) * n_pairs * n_splits;
    if (bal_nfull < 0) {
        if (n_units <= kMaxSchedUnits)
            build_dynamic_order(*t, BH, N, Nk, causal, head_block, n_pairs, n_splits);
    } else if (bal_nfull > 0)
        build_balanced_schedule(*t, static_cast<long long>(BH) * n_pairs, bal_nfull, grid, n_splits);
    else if (grid <= kMaxCtas && n_units <= kMaxSchedUnits)
        build_schedule(*t, BH, N, Nk, causal, head_block, n_pairs, n_splits, grid);
    if (g_sched_cache.size() >= 64)
        g_sched_cache.clear();
    g_sched_cache[key] = t;
    return t;
}

template <int D, bool SPLIT, int KIND>
cudaError_t launch_d(const FwdParams &p, int n_splits, float *opart, float *lpart, cudaStream_t stream,
                     unsigned int *status)
{
    using C = Cfg<D, elem_bytes<KIND>()>;
    const int BH = p.B * p.H;
    if (p.Hkv < 1 || p.H % p.Hkv != 0)
        return cudaErrorInvalidValue;
    const int BHkv = p.B * p.Hkv;
    CUtensorMap mq, mk, mv;
    if (!encode_map<D, KIND>(&mq, p.q, BH, p.N) || !encode_map<D, KIND>(&mk, p.k, BHkv, p.Nk) ||
        !encode_map<D, KIND>(&mv, p.v, BHkv, p.Nk))
        return cudaErrorInvalidValue;
    TcArgs a;
    a.p = p;
    a.n_pairs = (p.N + 2 * kBM - 1) / (2 * kBM);
    const long long units = static_cast<long long>(a.n_pairs) * BH * n_splits;
    if (units > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    a.n_units = static_cast<int>(units);
    a.head_block = head_block_for(BH, p.Nk, D, p.H / p.Hkv);
    a.n_splits = n_splits;
    a.opart = opart;
    a.lpart = lpart;
    a.status = status;
    int sms = 0;
    cudaError_t err = device_sm_count(&sms);
    if (err != cudaSuccess)
        return err;
    auto kernel = attn_fwd_tcgen05_kernel<D, SPLIT, KIND>;
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (err != cudaSuccess)
        return err;
    // The register split inside the kernel must fit the pool the CTA is launched with.
    cudaFuncAttributes fa;
    err = cudaFuncGetAttributes(&fa, kernel);
    if (err != cudaSuccess)
        return err;
    if (static_cast<long long>(fa.numRegs) * kThreads < RegSplit<D>::kPoolNeeded)
        return cudaErrorInvalidConfiguration;
    a.bal_chunks = 0;
    a.bal_nfull = 0;
    a.dynamic = 0;
    int grid = a.n_units < sms ? a.n_units : sms;
    if (SPLIT) {
        const int nf = splitkv_balanced_runs(BH, p.N, p.Nk, p.causal && !p.qrows, sms, n_splits);
        if (nf > 0) {
            const long long T = static_cast<long long>(a.n_pairs) * BH * nf;
            a.bal_nfull = nf;
            a.bal_chunks = static_cast<int>(T < sms ? T : sms);
            a.head_block = BH; // one head block: unit u is pair u / S, range u % S
            grid = a.bal_chunks;
        }
    }
    // Without balanced runs and with at least kDynamicUnitsPerSm units per SM, the units are dealt
    // dynamically: one CTA per unit, CTA c running unit unit[c] of the dynamic order
    // (build_dynamic_order; the unit order when the table does not fit), running CTAs taking
    // over the units of CTAs that have not started. Fewer units go to the static largest-first
    // table, which balances a short list better.
    std::shared_ptr<SchedTable> sched;
    if (a.bal_chunks == 0 && a.n_units >= kDynamicUnitsPerSm * sms) {
        a.dynamic = 1;
        grid = a.n_units;
        sched = schedule_for(BH, p.N, p.Nk, p.causal && !p.qrows, a.head_block, a.n_pairs, n_splits, grid, -1);
    } else {
        sched = schedule_for(BH, p.N, p.Nk, p.causal && !p.qrows, a.head_block, a.n_pairs, n_splits, grid,
                             a.bal_nfull);
    }
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
    err = cudaLaunchKernelEx(&cfg, kernel, a, mq, mk, mv, *sched);
    if (err != cudaSuccess)
        return err;
    return cudaGetLastError();
}

// Combination of the key ranges of split-KV for one row per warp, by the merge of two partial
// softmaxes of "Online Softmax Formulation" applied to S ranges at once: with lse_s the
// logsumexp of range s and O_s its normalised output, lse = log sum_s exp(lse_s) and
// O = sum_s exp(lse_s - lse) O_s. Ranges without an allowed key (lse_s = -inf) weigh 0; a
// row with none at all gets O = 0 and lse = -inf.
template <int D, int KIND>
__global__ void __launch_bounds__(256)
    attn_splitkv_merge_kernel(const float *__restrict__ opart, const float *__restrict__ lpart,
                              __half *__restrict__ o, float *__restrict__ lse, long long rows, int S)
{
    const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows)
        return;
    const float ls = lane < S ? lpart[static_cast<long long>(lane) * rows + row] : -INFINITY;
    float m = ls;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    const float ws = (m == -INFINITY || ls == -INFINITY) ? 0.f : expf(ls - m);
    float wsum = ws;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
    constexpr int kPer = D / 32; // output columns of this lane: [lane * kPer, lane * kPer + kPer)
    float acc[kPer];
#pragma unroll
    for (int c = 0; c < kPer; ++c)
        acc[c] = 0.f;
    for (int s = 0; s < S; ++s) {
        const float w = __shfl_sync(0xffffffffu, ws, s);
        if (w == 0.f)
            continue;
        const float *src = opart + (static_cast<long long>(s) * rows + row) * D + lane * kPer;
#pragma unroll
        for (int c = 0; c < kPer; ++c)
            acc[c] += w * src[c];
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    // O: fp32 for KIND tf32, else bf16 or fp16 rounded to nearest even
    const long long e0 = row * D + lane * kPer;
#pragma unroll
    for (int c = 0; c < kPer; ++c) {
        if constexpr (KIND == kKindTF32)
            reinterpret_cast<float *>(o)[e0 + c] = acc[c] * inv;
        else if constexpr (KIND == kKindBF16)
            reinterpret_cast<__nv_bfloat16 *>(o)[e0 + c] = __float2bfloat16_rn(acc[c] * inv);
        else
            o[e0 + c] = __float2half_rn(acc[c] * inv);
    }
    if (lse && lane == 0)
        lse[row] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
}

template <int D, int KIND>
cudaError_t launch_merge(const FwdParams &p, int n_splits, const float *opart, const float *lpart,
                         cudaStream_t stream)
{
    const long long rows = static_cast<long long>(p.B) * p.H * p.N;
    const long long blocks = (rows + 7) / 8;
    if (blocks > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    attn_splitkv_merge_kernel<D, KIND><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        opart, lpart, p.o, p.lse, rows, n_splits);
    return cudaGetLastError();
}

} // namespace

namespace {

template <int KIND>
cudaError_t launch_tcgen05_t(const FwdParams &p, cudaStream_t stream, unsigned int *status)
{
    if constexpr (KIND == kKindTF32) {
        // fp32 inputs: head dimension 32 only
        return p.d == 32 ? launch_d<32, false, KIND>(p, 1, nullptr, nullptr, stream, status)
                         : cudaErrorInvalidValue;
    } else {
        switch (p.d) {
        case 32: return launch_d<32, false, KIND>(p, 1, nullptr, nullptr, stream, status);
        case 64: return launch_d<64, false, KIND>(p, 1, nullptr, nullptr, stream, status);
        case 128: return launch_d<128, false, KIND>(p, 1, nullptr, nullptr, stream, status);
        default: return cudaErrorInvalidValue;
        }
    }
}

template <int KIND>
cudaError_t launch_splitkv_t(const FwdParams &p, int n_splits, float *opart, float *lpart,
                             cudaStream_t stream, unsigned int *status)
{
    cudaError_t err;
    if constexpr (KIND == kKindTF32) {
        if (p.d != 32)
            return cudaErrorInvalidValue;
        err = launch_d<32, true, KIND>(p, n_splits, opart, lpart, stream, status);
        if (err != cudaSuccess)
            return err;
        return launch_merge<32, KIND>(p, n_splits, opart, lpart, stream);
    } else {
        switch (p.d) {
        case 32: err = launch_d<32, true, KIND>(p, n_splits, opart, lpart, stream, status); break;
        case 64: err = launch_d<64, true, KIND>(p, n_splits, opart, lpart, stream, status); break;
        case 128: err = launch_d<128, true, KIND>(p, n_splits, opart, lpart, stream, status); break;
        default: return cudaErrorInvalidValue;
        }
        if (err != cudaSuccess)
            return err;
        switch (p.d) {
        case 32: return launch_merge<32, KIND>(p, n_splits, opart, lpart, stream);
        case 64: return launch_merge<64, KIND>(p, n_splits, opart, lpart, stream);
        default: return launch_merge<128, KIND>(p, n_splits, opart, lpart, stream);
        }
    }
}

} // namespace

int debug_schedule(int BH, int N, int Nk, int D, int G, int causal, int sms, int *units, int cap, int *off,
                   int *n_units, int *head_block)
{
    if (BH < 1 || N < 1 || Nk < 1 || G < 1 || sms < 1 || sms > kMaxCtas || (D != 32 && D != 64 && D != 128) ||
        (causal != 0 && causal != 1) || !units || !n_units || !head_block)
        return -1;
    const int n_pairs = (N + 2 * kBM - 1) / (2 * kBM);
    const long long nu = static_cast<long long>(BH) * n_pairs;
    if (nu > cap || nu > 0x7fffffffLL)
        return -1;
    const int hb = head_block_for(BH, Nk, D, G);
    *n_units = static_cast<int>(nu);
    *head_block = hb;
    // the same choice and tables as launch_d (one key range: no balanced split-KV runs)
    if (nu >= static_cast<long long>(kDynamicUnitsPerSm) * sms) {
        std::shared_ptr<SchedTable> t = schedule_for(BH, N, Nk, causal, hb, n_pairs, 1, static_cast<int>(nu), -1);
        for (int c = 0; c < nu; ++c)
            units[c] = t->use ? static_cast<int>(t->unit[c]) : c;
        return 1;
    }
    if (!off)
        return -1;
    const int grid = static_cast<int>(nu < sms ? nu : sms);
    std::shared_ptr<SchedTable> t = schedule_for(BH, N, Nk, causal, hb, n_pairs, 1, grid, 0);
    for (int c = 0; c <= grid; ++c)
        off[c] = t->use ? static_cast<int>(t->off[c]) : 0;
    for (int i = 0; t->use && i < off[grid]; ++i)
        units[i] = static_cast<int>(t->unit[i]);
    return 0;
}

cudaError_t launch_tcgen05(const FwdParams &p, cudaStream_t stream, unsigned int *status)
{
    switch (p.dtype) {
    case kDtypeF16: return launch_tcgen05_t<kKindF16>(p, stream, status);
    case kDtypeBF16: return launch_tcgen05_t<kKindBF16>(p, stream, status);
    case kDtypeF32: return launch_tcgen05_t<kKindTF32>(p, stream, status);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_tcgen05_splitkv(const FwdParams &p, int n_splits, float *opart, float *lpart,
                                   cudaStream_t stream, unsigned int *status)
{
    switch (p.dtype) {
    case kDtypeF16: return launch_splitkv_t<kKindF16>(p, n_splits, opart, lpart, stream, status);
    case kDtypeBF16: return launch_splitkv_t<kKindBF16>(p, n_splits, opart, lpart, stream, status);
    case kDtypeF32: return launch_splitkv_t<kKindTF32>(p, n_splits, opart, lpart, stream, status);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace attn
