// Internal interface between the C-ABI front end (attn_api.cu) and the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace attn {

// Element type of Q, K, V and O (the __half pointers below hold any of them).
constexpr int kDtypeF16 = 0;
constexpr int kDtypeBF16 = 1; // tcgen05 kernels only
constexpr int kDtypeF32 = 2;  // fp32 in and out, tf32 tensor-core products: tcgen05 kernel, d = 32

struct FwdParams {
    const __half *q;
    const __half *k;
    const __half *v;
    __half *o;
    int dtype;                  // kDtypeF16, kDtypeBF16 or kDtypeF32
    float *lse;                 // may be null
    const int32_t *key_lengths; // may be null
    int B, H, N, d; // N: query rows per head
    int Hkv, Nk;    // key/value heads per batch (H a multiple of Hkv) and keys per head;
                    // self-attention: Hkv = H, Nk = N. Query head h reads key/value head
                    // h / (H / Hkv); under the causal mask query i sees keys j <= i + Nk - N.
    int qrows;      // 0, or the query rows of one head when the rows of several query heads are
                    // packed into one problem (N = G * qrows, qrows < 128): under the causal
                    // mask row r is query r % qrows and sees keys j <= r % qrows + Nk - qrows.
    float sm_scale;
    float scale_log2; // sm_scale * log2(e): scores are exponentiated with exp2
    int causal;
    unsigned long long wait_limit_ns; // bound of every on-chip wait (nonzero)
    int inject_missing_arrive;        // self-test: withhold the first "P ready" arrival
};

// Default bound of an on-chip wait.
constexpr unsigned long long kDefaultWaitLimitNs = 4000000000ull;

// Warp-level mma.sync kernel (every d in {32, 64, 128}, every N).
cudaError_t launch_warp_mma(const FwdParams &p, cudaStream_t stream);

// TMA + tcgen05/TMEM kernel (d in {32, 64, 128}). `status` is the device status word.
cudaError_t launch_tcgen05(const FwdParams &p, cudaStream_t stream, unsigned int *status);

// Split-KV: the tcgen05 kernel over n_splits key ranges per (batch*head, Q tile pair), writing
// fp32 partial outputs opart [n_splits][B*H*N][d] and logsumexps lpart [n_splits][B*H*N], then
// the merge kernel writing o (and lse when non-null).
cudaError_t launch_tcgen05_splitkv(const FwdParams &p, int n_splits, float *opart, float *lpart,
                                   cudaStream_t stream, unsigned int *status);

// Balanced split-KV: when every (batch*head, Q tile pair) has the same K/V tile count (no
// causal mask, or a single pair), the tiles of all pairs are laid end to end and cut into one
// equal run per SM, each run one or two units; range s of a pair is its part of the s-th run
// that touches it. splitkv_balanced_runs: the per-pair tile count when a launch with n_splits
// ranges per pair uses these runs (they fit and finish sooner than equal ranges), else 0.
// splitkv_balanced_auto: the ranges per pair to ask for when balanced runs beat every equal
// split up to max_splits, else 0. (B*H, N and causal as the kernels run them.)
int splitkv_balanced_runs(int BH, int N, int Nk, int causal, int sms, int n_splits);
int splitkv_balanced_auto(int BH, int N, int Nk, int causal, int sms, int max_splits);

// Persistent short-sequence kernel (self-attention only: Nk = N <= 256, Hkv = H, d in {32, 64}).
cudaError_t launch_short(const FwdParams &p, cudaStream_t stream, unsigned int *status);

// fp32 inputs at fp32 accuracy (d = 32): split-TF32 products on the warp-level tensor core
// instruction, fp32 P and O.
cudaError_t launch_f32(const FwdParams &p, cudaStream_t stream);

// Naive three-pass forward (fp16 self-attention): S = sm_scale Q K^T into s ([B*H][N][Np] fp32),
// P = softmax(S + mask) into pm ([B*H][N][Np] fp16) with lse, then O = P V. Np =
// naive_padded_cols(N), N rounded up to a multiple of 128.
cudaError_t launch_naive(const FwdParams &p, float *s, __half *pm, cudaStream_t stream);
long long naive_padded_cols(int N);

// Decoding kernel (CUDA cores, no tensor cores): at most kDecodeMaxRows query rows per head
// (after query-group packing), fp16 or bf16, d in {32, 64, 128}, any key count. One
// thread-block cluster per head streams the head's keys and merges through distributed shared
// memory.
constexpr int kDecodeMaxRows = 16;
cudaError_t launch_decode(const FwdParams &p, cudaStream_t stream);

// Multiprocessor count of the current device (cached per device).
cudaError_t device_sm_count(int *out);

// The unit schedule the tiled kernel's host side builds for a launch of BH (batch * query head)
// problems of N query rows over Nk keys at head dimension D, G query heads per key/value head,
// on `sms` multiprocessors (one key range per Q-tile pair). Returns 1 for the dynamic schedule
// (units[c] = unit of CTA id c), 0 for the static table (CTA c's units at units[off[c] ..
// off[c + 1]); off has sms + 1 entries), -1 for bad arguments or a too small `cap`. n_units and
// head_block receive the unit count and the heads per L2 block.
int debug_schedule(int BH, int N, int Nk, int D, int G, int causal, int sms, int *units, int cap, int *off,
                   int *n_units, int *head_block);

// Status codes the kernels write into the device status word.
constexpr unsigned int kDevStatusTimeout = 1u;

} // namespace attn
