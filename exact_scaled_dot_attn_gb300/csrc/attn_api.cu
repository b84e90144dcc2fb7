// C-ABI front end: argument validation, kernel choice and launch.
// The operation and the contract of every entry point are stated in include/attn.h.
#include "attn.h"
#include "attn_internal.h"

#include <cmath>
#include <cstddef>
#include <cstdint>
#include <mutex>

extern "C" int attn_auto_path(int N, int d);

namespace {

// Per-device status word written by kernels whose bounded waits run out.
__device__ unsigned int g_attn_device_status;

constexpr int kMaxDevices = 64;
std::mutex g_status_mutex;
unsigned int *g_status_ptr[kMaxDevices];

// Device address of the status word for the current device (looked up once per device).
cudaError_t status_word(unsigned int **out)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_status_mutex);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_attn_device_status);
        if (err != cudaSuccess)
            return err;
        g_status_ptr[dev] = static_cast<unsigned int *>(p);
    }
    *out = g_status_ptr[dev];
    return cudaSuccess;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Sizes of one call: H query heads of N_q rows, H_kv key/value heads of N_k keys.
struct Shape {
    int B, H, Hkv, Nq, Nk, d;
    int dtype;     // attn_dtype_t
    int qrows = 0; // packed query groups under the causal mask: query rows of one head
    bool self() const { return Hkv == H && Nq == Nk && qrows == 0; }
};

attn_status_t validate(const void *q, const void *k, const void *v, const void *o, const float *lse,
                       const Shape &sh, float sm_scale, int causal, const int32_t *key_lengths)
{
    if (!q || !k || !v || !o)
        return ATTN_ERR_INVALID_ARG;
    if (sh.B < 1 || sh.H < 1 || sh.Hkv < 1 || sh.Nq < 1 || sh.Nk < 1 || sh.H % sh.Hkv != 0)
        return ATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1)
        return ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(sm_scale))
        return ATTN_ERR_INVALID_ARG;
    if (sh.d != 32 && sh.d != 64 && sh.d != 128)
        return ATTN_ERR_UNSUPPORTED;
    if (sh.dtype != ATTN_DTYPE_F16 && sh.dtype != ATTN_DTYPE_BF16 && sh.dtype != ATTN_DTYPE_F32)
        return ATTN_ERR_UNSUPPORTED;
    if (sh.dtype == ATTN_DTYPE_F32 && sh.d != 32) // fp32 inputs: head dimension 32 only
        return ATTN_ERR_UNSUPPORTED;
    const int64_t bh = static_cast<int64_t>(sh.B) * sh.H;
    if (bh > INT32_MAX)
        return ATTN_ERR_INVALID_ARG;
    const int64_t bhkv = static_cast<int64_t>(sh.B) * sh.Hkv;
    // element count of every tensor must fit int64
    if (bh * sh.Nq > INT64_MAX / sh.d || bhkv * sh.Nk > INT64_MAX / sh.d)
        return ATTN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
        return ATTN_ERR_MISALIGNED;
    if ((lse && !aligned(lse, 4)) || (key_lengths && !aligned(key_lengths, 4)))
        return ATTN_ERR_MISALIGNED;
    return ATTN_OK;
}

attn::FwdParams make_params(const void *q, const void *k, const void *v, void *o, float *lse,
                            const Shape &sh, float sm_scale, int causal, const int32_t *key_lengths)
{
    attn::FwdParams p;
    p.q = static_cast<const __half *>(q);
    p.k = static_cast<const __half *>(k);
    p.v = static_cast<const __half *>(v);
    p.o = static_cast<__half *>(o);
    p.lse = lse;
    p.key_lengths = key_lengths;
    p.B = sh.B;
    p.H = sh.H;
    p.N = sh.Nq;
    p.d = sh.d;
    p.Hkv = sh.Hkv;
    p.Nk = sh.Nk;
    p.qrows = sh.qrows;
    p.dtype = sh.dtype == ATTN_DTYPE_BF16 ? attn::kDtypeBF16
              : sh.dtype == ATTN_DTYPE_F32 ? attn::kDtypeF32
                                           : attn::kDtypeF16;
    p.sm_scale = sm_scale;
    p.scale_log2 = sm_scale * 1.4426950408889634f;
    p.causal = causal;
    p.wait_limit_ns = attn::kDefaultWaitLimitNs;
    p.inject_missing_arrive = 0;
    return p;
}

Shape self_shape(int B, int H, int N, int d) { return Shape{B, H, H, N, N, d, ATTN_DTYPE_F16}; }

// Grouped-query attention with few query rows: the G = H / H_kv query heads that share a
// key/value head are adjacent in Q, O and lse ([B, H, N_q, d] = [B, H_kv, G * N_q, d]), so the
// problem is the same attention with H_kv heads of G * N_q query rows each, and the rows of a
// group fill one Q tile together. Without the causal mask every row keeps its keys; with it
// and one query row, query 0 sees every key (j <= N_k - 1), so the mask goes; with it and more
// rows, the kernels take row r as query r % N_q (qrows). Applied below 128 query rows, where a
// head alone would leave a tile mostly empty.
void pack_query_groups(Shape &sh, int &causal)
{
    if (sh.Hkv < sh.H && sh.Nq < 128) {
        const long long rows = static_cast<long long>(sh.H / sh.Hkv) * sh.Nq;
        if (rows <= INT32_MAX) {
            if (causal && sh.Nq > 1)
                sh.qrows = sh.Nq;
            else
                causal = 0;
            sh.Nq = static_cast<int>(rows);
            sh.H = sh.Hkv;
        }
    }
}

// The decoding kernel takes fp16 and bf16 problems of at most kDecodeMaxRows rows per head
// (counted after packing).
bool decode_fits(const Shape &sh) { return sh.dtype != ATTN_DTYPE_F32 && sh.Nq <= attn::kDecodeMaxRows; }

// The kernel ATTN_PATH_AUTO runs for a (packed) shape.
int auto_choice(const Shape &sh)
{
    if (decode_fits(sh) && sh.Nk >= ATTN_DECODE_MIN_KEYS)
        return ATTN_PATH_DECODE; // a few rows over many keys: bound by reading K and V
    if (sh.dtype == ATTN_DTYPE_F32)
        return ATTN_PATH_WARP_MMA; // fp32 accuracy
    if (sh.self() && sh.dtype == ATTN_DTYPE_F16)
        return attn_auto_path(sh.Nq, sh.d);
    return ATTN_PATH_TCGEN05;
}

// One forward pass on the chosen kernel (the automatic choice when path is ATTN_PATH_AUTO).
attn_status_t run_fwd(const void *q, const void *k, const void *v, void *o, float *lse, const Shape &sh_in,
                      float sm_scale, int causal_in, const int32_t *key_lengths, int path,
                      const attn_debug_opts_t *opts, attn_stream_t stream);

} // namespace

extern "C" const char *attn_status_str(attn_status_t status)
{
    switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported head dimension or path";
    case ATTN_ERR_MISALIGNED: return "tensor pointer not 16-byte aligned";
    case ATTN_ERR_CUDA: return "CUDA call failed";
    case ATTN_ERR_TIMEOUT: return "bounded on-chip wait ran out";
    case ATTN_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the fixed no-allocation array holds";
    default: return "unknown status";
    }
}

extern "C" int attn_auto_path(int N, int d)
{
    if (d != 32 && d != 64 && d != 128)
        return -1;
    // Head dimension 32 with at most 256 keys: the short-sequence kernel (a whole score row
    // per Q tile in Tensor Memory); everything else: the tiled tcgen05 kernel.
    if (d == 32 && N <= 256)
        return ATTN_PATH_SHORT;
    return ATTN_PATH_TCGEN05;
}

namespace {

attn_status_t run_fwd(const void *q, const void *k, const void *v, void *o, float *lse, const Shape &sh_in,
                      float sm_scale, int causal_in, const int32_t *key_lengths, int path,
                      const attn_debug_opts_t *opts, attn_stream_t stream)
{
    attn_status_t st = validate(q, k, v, o, lse, sh_in, sm_scale, causal_in, key_lengths);
    if (st != ATTN_OK)
        return st;
    if (path != ATTN_PATH_AUTO && path != ATTN_PATH_WARP_MMA && path != ATTN_PATH_TCGEN05 &&
        path != ATTN_PATH_SHORT && path != ATTN_PATH_DECODE)
        return ATTN_ERR_UNSUPPORTED;
    // an explicitly chosen short-sequence kernel takes only the shapes the caller gave it
    if (path == ATTN_PATH_SHORT && !sh_in.self())
        return ATTN_ERR_UNSUPPORTED;
    Shape sh = sh_in;
    int causal = causal_in;
    pack_query_groups(sh, causal);
    // The short-sequence kernel serves fp16 self-attention only; bf16 and fp32 run on the
    // tiled tcgen05 kernel only.
    if (path == ATTN_PATH_SHORT && (!sh.self() || sh.Nq > 256 || sh.d > 64))
        return ATTN_ERR_UNSUPPORTED;
    if (path == ATTN_PATH_DECODE && !decode_fits(sh))
        return ATTN_ERR_UNSUPPORTED;
    // bf16 runs on the tcgen05 and decoding kernels only; fp32 on the tcgen05 kernel (TF32
    // products) or on the warp-level kernel (split-TF32 products, fp32 accuracy)
    if (sh.dtype == ATTN_DTYPE_BF16 && path != ATTN_PATH_AUTO && path != ATTN_PATH_TCGEN05 &&
        path != ATTN_PATH_DECODE)
        return ATTN_ERR_UNSUPPORTED;
    if (sh.dtype == ATTN_DTYPE_F32 && path == ATTN_PATH_SHORT)
        return ATTN_ERR_UNSUPPORTED;
    if (path == ATTN_PATH_AUTO)
        path = auto_choice(sh);

    attn::FwdParams p = make_params(q, k, v, o, lse, sh, sm_scale, causal, key_lengths);
    if (opts && opts->wait_limit_ns)
        p.wait_limit_ns = opts->wait_limit_ns;
    p.inject_missing_arrive = opts ? (opts->inject_missing_arrive != 0) : 0;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t err;
    if (path == ATTN_PATH_DECODE) {
        err = attn::launch_decode(p, s);
    } else if (path == ATTN_PATH_TCGEN05 || path == ATTN_PATH_SHORT) {
        unsigned int *status = nullptr;
        err = status_word(&status);
        if (err == cudaSuccess)
            err = path == ATTN_PATH_TCGEN05 ? attn::launch_tcgen05(p, s, status)
                                            : attn::launch_short(p, s, status);
    } else {
        err = sh.dtype == ATTN_DTYPE_F32 ? attn::launch_f32(p, s) : attn::launch_warp_mma(p, s);
    }
    return err == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

} // namespace

extern "C" int attn_auto_path_ex(int H, int H_kv, int N_q, int N_k, int d, int dtype, int causal)
{
    if (H < 1 || H_kv < 1 || H % H_kv != 0 || N_q < 1 || N_k < 1 || (d != 32 && d != 64 && d != 128) ||
        (dtype != ATTN_DTYPE_F16 && dtype != ATTN_DTYPE_BF16 && dtype != ATTN_DTYPE_F32) ||
        (dtype == ATTN_DTYPE_F32 && d != 32) || (causal != 0 && causal != 1))
        return -1;
    Shape sh{1, H, H_kv, N_q, N_k, d, dtype};
    pack_query_groups(sh, causal);
    return auto_choice(sh);
}

extern "C" int attn_debug_schedule(int BH, int N_q, int N_k, int d, int G, int causal, int sms, int *units,
                                   int units_cap, int *off, int *n_units, int *head_block)
{
    return attn::debug_schedule(BH, N_q, N_k, d, G, causal, sms, units, units_cap, off, n_units, head_block);
}

extern "C" attn_status_t attn_fwd_debug(const void *q, const void *k, const void *v, void *o,
                                        float *lse, int B, int H, int N, int d, float sm_scale,
                                        int causal, const int32_t *key_lengths, int path,
                                        const attn_debug_opts_t *opts, attn_stream_t stream)
{
    return run_fwd(q, k, v, o, lse, self_shape(B, H, N, d), sm_scale, causal, key_lengths, path, opts,
                   stream);
}

extern "C" attn_status_t attn_fwd_ex(const void *q, const void *k, const void *v, void *o, float *lse,
                                     int B, int H, int H_kv, int N_q, int N_k, int d, int dtype,
                                     float sm_scale, int causal, const int32_t *key_lengths, int path,
                                     attn_stream_t stream)
{
    return run_fwd(q, k, v, o, lse, Shape{B, H, H_kv, N_q, N_k, d, dtype}, sm_scale, causal, key_lengths,
                   path, nullptr, stream);
}

extern "C" attn_status_t attn_fwd_path(const void *q, const void *k, const void *v, void *o,
                                       float *lse, int B, int H, int N, int d, float sm_scale,
                                       int causal, const int32_t *key_lengths, int path,
                                       attn_stream_t stream)
{
    return attn_fwd_debug(q, k, v, o, lse, B, H, N, d, sm_scale, causal, key_lengths, path, nullptr,
                          stream);
}

extern "C" attn_status_t attn_fwd_lse(const void *q, const void *k, const void *v, void *o,
                                      float *lse, int B, int H, int N, int d, float sm_scale,
                                      int causal, const int32_t *key_lengths, attn_stream_t stream)
{
    return attn_fwd_path(q, k, v, o, lse, B, H, N, d, sm_scale, causal, key_lengths,
                         ATTN_PATH_AUTO, stream);
}

extern "C" attn_status_t attn_fwd(const void *q, const void *k, const void *v, void *o, int B,
                                  int H, int N, int d, float sm_scale, int causal,
                                  const int32_t *key_lengths, attn_stream_t stream)
{
    return attn_fwd_path(q, k, v, o, nullptr, B, H, N, d, sm_scale, causal, key_lengths,
                         ATTN_PATH_AUTO, stream);
}

namespace {

constexpr int kMaxSplits = 16;

// Bytes of split-KV workspace: fp32 partial outputs [S][B*H*N][d] then logsumexps [S][B*H*N];
// 0 when the sizes are invalid or the byte count does not fit size_t.
size_t splitkv_bytes(int B, int H, int N, int d, int S)
{
    if (B < 1 || H < 1 || N < 1 || (d != 32 && d != 64 && d != 128) || S < 1 || S > kMaxSplits)
        return 0;
    const unsigned long long rows = static_cast<unsigned long long>(B) * H * N;
    const unsigned long long per = rows * (static_cast<unsigned long long>(d) + 1) * 4ull;
    if (rows == 0 || per / rows / 4ull != static_cast<unsigned long long>(d) + 1)
        return 0;
    const unsigned long long total = per * static_cast<unsigned long long>(S);
    if (total / static_cast<unsigned long long>(S) != per || total > static_cast<unsigned long long>(SIZE_MAX))
        return 0;
    return static_cast<size_t>(total);
}

// Ranges per (batch*head, Q tile pair) for the automatic choice. When every pair has the same
// K/V tile count and balanced runs over all pairs finish sooner than any equal split, the
// ranges those runs need (attn::splitkv_balanced_auto). Otherwise: without the causal mask every
// (pair, range) unit has the same length, so the most ranges that still give one unit per SM
// (floor(SMs / pairs)) shorten the launch without adding a second wave. With it, enough units
// that the largest is no longer than an SM's average share: the largest pair's K/V tile count
// over the mean (about 2 for self-attention; from the shifted diagonal for cross-attention)
// times SMs / pairs, rounded up. At most one range per two K/V tiles, at most kMaxSplits.
int auto_splits(int B, int H, int Nq, int Nk, int causal, int sms)
{
    // balanced runs over all pairs, where they finish sooner than any equal split
    const int bal = attn::splitkv_balanced_auto(B * H, Nq, Nk, causal, sms, kMaxSplits);
    if (bal > 0)
        return bal;
    const int n_pairs = (Nq + 255) / 256;
    const long long pairs = static_cast<long long>(B) * H * n_pairs;
    long long want;
    if (!causal) {
        want = sms / pairs;
    } else {
        long long sum = 0, mx = 0;
        for (int pr = 0; pr < n_pairs; ++pr) {
            long long e = static_cast<long long>(pr) * 256 + 256 + Nk - Nq;
            e = e < 0 ? 0 : (e > Nk ? Nk : e);
            const long long f = (e + 127) / 128;
            sum += f;
            mx = f > mx ? f : mx;
        }
        const double skew = sum > 0 ? static_cast<double>(mx) * n_pairs / static_cast<double>(sum) : 1.0;
        want = static_cast<long long>(std::ceil(static_cast<double>(sms) * skew / pairs));
    }
    const int kv_tiles = (Nk + 127) / 128;
    long long s = want < 1 ? 1 : want;
    if (s > kv_tiles / 2)
        s = kv_tiles / 2;
    if (s > kMaxSplits)
        s = kMaxSplits;
    return s < 1 ? 1 : static_cast<int>(s);
}

} // namespace

extern "C" size_t attn_splitkv_workspace_bytes(int B, int H, int N, int d, int n_splits)
{
    return splitkv_bytes(B, H, N, d, n_splits);
}

extern "C" int attn_splitkv_auto_splits_ex(int B, int H, int H_kv, int N_q, int N_k, int d, int causal)
{
    if (B < 1 || H < 1 || H_kv < 1 || H % H_kv != 0 || N_q < 1 || N_k < 1 ||
        (d != 32 && d != 64 && d != 128) || (causal != 0 && causal != 1))
        return -1;
    int sms = 0;
    if (attn::device_sm_count(&sms) != cudaSuccess || sms < 1)
        sms = 152; // GB300's count, for a query made where no device answers
    // the shape the kernels run (query heads of a group packed together, see pack_query_groups)
    Shape sh{B, H, H_kv, N_q, N_k, d, ATTN_DTYPE_F16};
    pack_query_groups(sh, causal);
    // packed groups under the causal mask: every pair sees all keys, as without the mask
    return auto_splits(sh.B, sh.H, sh.Nq, sh.Nk, sh.qrows ? 0 : causal, sms);
}

extern "C" int attn_splitkv_auto_splits(int B, int H, int N, int d, int causal)
{
    return attn_splitkv_auto_splits_ex(B, H, H, N, N, d, causal);
}

extern "C" attn_status_t attn_fwd_splitkv_ex(const void *q, const void *k, const void *v, void *o,
                                             float *lse, int B, int H, int H_kv, int N_q, int N_k, int d,
                                             int dtype, float sm_scale, int causal,
                                             const int32_t *key_lengths, int n_splits, void *workspace,
                                             size_t workspace_bytes, attn_stream_t stream)
{
    Shape sh{B, H, H_kv, N_q, N_k, d, dtype};
    attn_status_t st = validate(q, k, v, o, lse, sh, sm_scale, causal, key_lengths);
    if (st != ATTN_OK)
        return st;
    if (n_splits <= 0) {
        n_splits = attn_splitkv_auto_splits_ex(B, H, H_kv, N_q, N_k, d, causal);
        if (n_splits < 1)
            return ATTN_ERR_INVALID_ARG;
    }
    // (the workspace holds one partial row per query row: B * H * N_q either way)
    pack_query_groups(sh, causal);
    if (n_splits > kMaxSplits)
        return ATTN_ERR_INVALID_ARG;
    const size_t need = splitkv_bytes(B, H, N_q, d, n_splits);
    if (need == 0 || !workspace || workspace_bytes < need)
        return ATTN_ERR_INVALID_ARG;
    if (!aligned(workspace, 16))
        return ATTN_ERR_MISALIGNED;
    attn::FwdParams p = make_params(q, k, v, o, lse, sh, sm_scale, causal, key_lengths);
    unsigned int *status = nullptr;
    cudaError_t err = status_word(&status);
    if (err != cudaSuccess)
        return ATTN_ERR_CUDA;
    float *opart = static_cast<float *>(workspace);
    float *lpart = opart + static_cast<size_t>(n_splits) * B * H * N_q * d;
    err = attn::launch_tcgen05_splitkv(p, n_splits, opart, lpart, reinterpret_cast<cudaStream_t>(stream),
                                       status);
    return err == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

extern "C" attn_status_t attn_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                                          int B, int H, int N, int d, float sm_scale, int causal,
                                          const int32_t *key_lengths, int n_splits, void *workspace,
                                          size_t workspace_bytes, attn_stream_t stream)
{
    return attn_fwd_splitkv_ex(q, k, v, o, lse, B, H, H, N, N, d, ATTN_DTYPE_F16, sm_scale, causal,
                               key_lengths, n_splits, workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------- naive three-pass baseline
namespace {

// Bytes of the naive pass's workspace: S [B*H][N][Np] fp32, then P [B*H][N][Np] fp16; 0 when
// the sizes are invalid or the count does not fit size_t.
size_t naive_bytes(int B, int H, int N)
{
    if (B < 1 || H < 1 || N < 1)
        return 0;
    const unsigned long long rows = static_cast<unsigned long long>(B) * H * N;
    const unsigned long long np = static_cast<unsigned long long>(attn::naive_padded_cols(N));
    if (rows > (1ull << 40) || np > (1ull << 32))
        return 0;
    const unsigned long long elems = rows * np;
    if (elems / np != rows || elems > static_cast<unsigned long long>(SIZE_MAX) / 6ull)
        return 0;
    return static_cast<size_t>(elems * 6ull);
}

} // namespace

extern "C" size_t attn_naive_workspace_bytes(int B, int H, int N) { return naive_bytes(B, H, N); }

extern "C" attn_status_t attn_fwd_naive(const void *q, const void *k, const void *v, void *o, float *lse,
                                        int B, int H, int N, int d, float sm_scale, int causal,
                                        const int32_t *key_lengths, void *workspace,
                                        size_t workspace_bytes, attn_stream_t stream)
{
    attn_status_t st = validate(q, k, v, o, lse, self_shape(B, H, N, d), sm_scale, causal, key_lengths);
    if (st != ATTN_OK)
        return st;
    const size_t need = naive_bytes(B, H, N);
    if (need == 0 || !workspace || workspace_bytes < need)
        return ATTN_ERR_INVALID_ARG;
    if (!aligned(workspace, 16))
        return ATTN_ERR_MISALIGNED;
    attn::FwdParams p = make_params(q, k, v, o, lse, self_shape(B, H, N, d), sm_scale, causal, key_lengths);
    float *s = static_cast<float *>(workspace);
    __half *pm = reinterpret_cast<__half *>(s + static_cast<size_t>(B) * H * N * attn::naive_padded_cols(N));
    const cudaError_t err = attn::launch_naive(p, s, pm, reinterpret_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// ---------------------------------------------------------------- split-KV without allocation
//
// Some callers cannot allocate device memory on the path that calls the attention: a serving
// process whose device memory is already handed out to its own pool or caching allocator (a
// cudaMalloc there fails, or takes memory the pool counted on), a plug-in running inside
// another runtime that gives it no allocator, or a latency-bound request loop where the
// implicit synchronisation of cudaMalloc/cudaFree is not acceptable. For them the split-KV
// forward can run on a fixed scratch array that is part of this library's device image: the
// caller passes only inputs and outputs.
namespace {

// The scratch array (fp32 partial outputs, then partial logsumexps). Every GPU on which the
// library's device code is loaded holds it until the process exits.
constexpr size_t kNoAllocScratchBytes = 64ull << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mutex;
void *g_noalloc_ptr[kMaxDevices];

// Device address of the scratch array on the current device, looked up once per device with
// that device current.
cudaError_t noalloc_scratch(void **out)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (err != cudaSuccess)
            return err;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}

} // namespace

extern "C" size_t attn_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" attn_status_t attn_fwd_splitkv_noalloc(const void *q, const void *k, const void *v, void *o,
                                                  float *lse, int B, int H, int N, int d, float sm_scale,
                                                  int causal, const int32_t *key_lengths, int n_splits,
                                                  attn_stream_t stream)
{
    attn_status_t st = validate(q, k, v, o, lse, self_shape(B, H, N, d), sm_scale, causal, key_lengths);
    if (st != ATTN_OK)
        return st;
    if (n_splits <= 0) {
        n_splits = attn_splitkv_auto_splits(B, H, N, d, causal);
        if (n_splits < 1)
            return ATTN_ERR_INVALID_ARG;
        // the automatic count, lowered to the most ranges whose partials fit the array
        while (n_splits > 1 && splitkv_bytes(B, H, N, d, n_splits) > kNoAllocScratchBytes)
            --n_splits;
    }
    if (n_splits > kMaxSplits)
        return ATTN_ERR_INVALID_ARG;
    const size_t need = splitkv_bytes(B, H, N, d, n_splits);
    if (need == 0)
        return ATTN_ERR_INVALID_ARG;
    if (need > kNoAllocScratchBytes)
        return ATTN_ERR_SCRATCH_LIMIT;
    void *scratch = nullptr;
    if (noalloc_scratch(&scratch) != cudaSuccess)
        return ATTN_ERR_CUDA;
    // Nothing in the array needs clearing: the split kernel writes every partial output and
    // logsumexp the merge reads, in this call.
    return attn_fwd_splitkv(q, k, v, o, lse, B, H, N, d, sm_scale, causal, key_lengths, n_splits, scratch,
                            kNoAllocScratchBytes, stream);
}

extern "C" attn_status_t attn_read_device_status(attn_stream_t stream)
{
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    unsigned int value = 0;
    if (cudaMemcpyFromSymbol(&value, g_attn_device_status, sizeof(value)) != cudaSuccess)
        return ATTN_ERR_CUDA;
    if (value != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_attn_device_status, &zero, sizeof(zero)) != cudaSuccess)
            return ATTN_ERR_CUDA;
        return ATTN_ERR_TIMEOUT;
    }
    return ATTN_OK;
}
