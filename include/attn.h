/*
 * attn.h -- C ABI of the GB300 (sm_103a) exact scaled dot-product attention forward.
 *
 * The operation, for every batch b, head h and query row i of a self-attention
 * problem with N queries and N keys per head:
 *
 *     O_i = sum_j softmax_j( sm_scale * q_i . k_j + mask_ij ) v_j
 *
 * ("Tensor Parallelism with CUDA - Standard Attention", sections "Step 1: QK^T",
 * "Step 2: Softmax" and "Step 3: PV"; the additive mask of "Naive Attention
 * Kernel", section "1. Standard Attention: Step by Step", restricted to the two
 * structured masks below). The kernels follow the tiled recurrence of
 * "Self-Attention Kernel & Inference Engine from Scratch", sections "Online
 * Softmax Formulation" and "CUDA Kernel Structure": Q, K and V tiles are staged
 * on chip and the N x N score matrix is never written to memory.
 *
 * Masks (mask_ij is 0 or -inf):
 *   causal        key j is allowed for query i only when j <= i (square, top-left aligned);
 *   key_lengths   key j of batch b is allowed only when j < clamp(key_lengths[b], 0, N)
 *                 (the key-padding mask of the "cuda-reranker" README). Padded query rows
 *                 (i >= key_lengths[b]) are computed like any other row.
 *   A row whose allowed set is empty gets O_i = 0 and lse_i = -inf.
 *
 * Data layout and types (all tensors contiguous, d innermost):
 *   q, k, v   fp16 (IEEE binary16) [B, H, N, d], device memory
 *   o         fp16 [B, H, N, d], device memory, written (rounded to nearest even)
 *   lse       fp32 [B, H, N] natural-log logsumexp of the scaled allowed scores, or NULL
 *   key_lengths  int32 [B] in device memory, or NULL (= N for every batch)
 * Arithmetic: fp16 products, fp32 accumulation, fp32 row statistics; the
 * probabilities are rounded to fp16 before the PV product.
 *
 * Ownership: the caller owns every buffer. The entry points allocate no memory,
 * keep no per-call state and are safe to call from several host threads, with one
 * exception: attn_fwd_splitkv_noalloc shares one fixed scratch array per GPU among all
 * its calls, and its declaration states how such calls must be ordered.
 *
 * Errors: argument errors are returned synchronously, before anything is
 * launched. Launch failures return ATTN_ERR_CUDA. The work is asynchronous on
 * `stream` (NULL = the legacy default stream) and the call does not
 * synchronize; device-side faults surface at the caller's next synchronizing
 * CUDA call. Kernels that wait on on-chip barriers bound every wait; a wait that
 * runs out ends the block early and records ATTN_ERR_TIMEOUT in a per-device
 * status word that attn_read_device_status() returns.
 *
 * Stream order: the tiled and short-sequence kernels use programmatic dependent launch.
 * Their set-up (barrier initialisation, Tensor Memory allocation) may overlap the end of
 * the previous kernel on the stream, but they read and write no global memory before that
 * kernel has completed. Ordering against earlier work is therefore that of an ordinary
 * launch. They also let the next kernel on the stream start early. A kernel that the
 * caller launches right after them with programmatic stream serialization must call
 * cudaGridDependencySynchronize() (griddepcontrol.wait) before it reads O or lse.
 * Ordinary launches need nothing.
 */
#ifndef ATTN_GB300_ATTN_H
#define ATTN_GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without pulling in the CUDA headers. */
typedef struct CUstream_st *attn_stream_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1, /* NULL tensor pointer, B/H/N < 1, non-finite sm_scale, size overflow */
    ATTN_ERR_UNSUPPORTED = 2, /* head dimension other than 32, 64 or 128; unknown path */
    ATTN_ERR_MISALIGNED = 3,  /* a tensor pointer that is not 16-byte aligned */
    ATTN_ERR_CUDA = 4,        /* a CUDA runtime or driver call failed */
    ATTN_ERR_TIMEOUT = 5,     /* a bounded on-chip wait ran out (see attn_read_device_status) */
    ATTN_ERR_SCRATCH_LIMIT = 6 /* attn_fwd_splitkv_noalloc: the problem needs more scratch than
                                  attn_noalloc_scratch_bytes() */
} attn_status_t;

/* Element type of Q, K, V and O for attn_fwd_ex / attn_fwd_splitkv_ex (the other entry points
 * take fp16). bf16 (8-bit exponent, 8-bit significand) runs on the tiled tcgen05 kernel only,
 * with P rounded to bf16 as well: one tcgen05 MMA takes A and B of the same type. fp32 (the
 * "cuda-reranker" README's precision, on the tensor cores that README names as its next step)
 * takes fp32 Q, K, V and writes fp32 O, d = 32 only, in one of two ways:
 *   - ATTN_PATH_AUTO or ATTN_PATH_WARP_MMA: fp32 accuracy. Every operand of both products, P
 *     included, is split into a TF32 part and a TF32 remainder and each product is formed from
 *     three TF32 products (error-corrected TF32, Ootomo and Yokota 2022): products within about
 *     2^-21 of their fp32 value, fp32 accumulation, P never rounded below fp32. Warp-level
 *     tensor-core kernel (mma.sync m16n8k8 tf32).
 *   - ATTN_PATH_TCGEN05 (and attn_fwd_splitkv_ex): TF32 products, the tensor core using the
 *     sign, the exponent and the 10 leading fraction bits of each fp32 operand, P included;
 *     fp32 accumulation and softmax statistics. Faster, at TF32's precision. */
typedef enum {
    ATTN_DTYPE_F16 = 0,
    ATTN_DTYPE_BF16 = 1,
    ATTN_DTYPE_F32 = 2
} attn_dtype_t;

/* Which kernel runs the forward. AUTO runs the decoding kernel for problems of at most 16
 * query rows per head (after the query-group packing of attn_fwd_ex) over at least
 * ATTN_DECODE_MIN_KEYS keys in fp16 or bf16, the short-sequence kernel for fp16
 * self-attention with d = 32 and N <= 256, the warp-level split-TF32 kernel for fp32 inputs
 * (fp32 accuracy), and the tiled tcgen05 kernel everywhere else (the fastest at every measured
 * shape); the other kernels remain selectable explicitly. */
typedef enum {
    ATTN_PATH_AUTO = 0,
    ATTN_PATH_WARP_MMA = 1, /* warp-level mma.sync tile kernel: every d, every N */
    ATTN_PATH_TCGEN05 = 2,  /* TMA + tcgen05/TMEM warp-specialised tiled kernel: every d, every N */
    ATTN_PATH_SHORT = 3,    /* tcgen05 kernel holding a Q tile's whole score row in TMEM
                               (two CTAs per SM, heads dealt longest first): N <= 256,
                               d in {32, 64} */
    ATTN_PATH_DECODE = 4    /* decoding kernel on the CUDA cores, K and V streamed once through
                               shared memory by thread-block clusters that merge a head's key
                               ranges in distributed shared memory: at most 16 query rows per
                               head (counted after query-group packing), fp16 or bf16, any N_k */
} attn_path_t;

/* Fewest keys for which ATTN_PATH_AUTO takes the decoding kernel. */
#define ATTN_DECODE_MIN_KEYS 256

/*
 * Forward without logsumexp. Arguments as described above:
 *   q, k, v, o   device pointers, 16-byte aligned, fp16 [B,H,N,d]
 *   B, H, N      >= 1; B*H*N*d must fit in int64 and B*H in int32
 *   d            32, 64 or 128 (the head dimensions of the "CUDA Kernel Structure" template)
 *   sm_scale     finite; 1/sqrt(d) is the usual choice ("Why Divide by sqrt(d)?")
 *   causal       0 or 1
 *   key_lengths  device int32 [B] or NULL
 *   stream       CUDA stream or NULL
 */
attn_status_t attn_fwd(const void *q, const void *k, const void *v, void *o, int B, int H, int N,
                       int d, float sm_scale, int causal, const int32_t *key_lengths,
                       attn_stream_t stream);

/* Forward that also writes lse (fp32 [B,H,N], device, 4-byte aligned) when lse != NULL. */
attn_status_t attn_fwd_lse(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                           int H, int N, int d, float sm_scale, int causal,
                           const int32_t *key_lengths, attn_stream_t stream);

/* attn_fwd_lse with an explicit kernel choice (attn_path_t). A kernel asked for a
 * shape it does not take (ATTN_PATH_SHORT with N > 256 or d = 128, ATTN_PATH_DECODE with
 * N > 16) returns ATTN_ERR_UNSUPPORTED. Used to check each kernel on every shape it serves. */
attn_status_t attn_fwd_path(const void *q, const void *k, const void *v, void *o, float *lse,
                            int B, int H, int N, int d, float sm_scale, int causal,
                            const int32_t *key_lengths, int path, attn_stream_t stream);

/* Test hooks of attn_fwd_debug (the pages have no counterpart: these exercise the
 * library's own bounded waits). */
typedef struct {
    uint64_t wait_limit_ns;    /* bound of every on-chip wait; 0 = the default, 4 s */
    int inject_missing_arrive; /* 1: the softmax warps of the tcgen05 kernel withhold their
                                  first "P ready" arrival of every unit, so the MMA warp's
                                  bounded wait runs out and the kernel records
                                  ATTN_ERR_TIMEOUT (outputs are then undefined); 0 in use */
} attn_debug_opts_t;

/* attn_fwd_path with test hooks (opts may be NULL = defaults). Used by the self-test of
 * the timeout path: the launch returns ATTN_OK, and attn_read_device_status() then
 * reports ATTN_ERR_TIMEOUT while the context stays usable. */
attn_status_t attn_fwd_debug(const void *q, const void *k, const void *v, void *o, float *lse,
                             int B, int H, int N, int d, float sm_scale, int causal,
                             const int32_t *key_lengths, int path, const attn_debug_opts_t *opts,
                             attn_stream_t stream);

/* Test hook: the unit schedule of the tiled kernel for a launch of BH = B * H query-head
 * problems of N_q rows over N_k keys at head dimension d, G = H / H_kv query heads per key/value
 * head, on `sms` multiprocessors (1 <= sms <= 256), one key range per Q-tile pair (a unit is a
 * (batch * head, pair of 128-row Q tiles)). Host computation only: no device is touched.
 * Returns 1 for the dynamic schedule (one CTA per unit; units[c] is the unit of CTA id c),
 * 0 for the static table (a persistent grid of min(units, sms) CTAs; CTA c's units, in order,
 * are units[off[c] .. off[c + 1]), off holding sms + 1 entries; all off zero when the table
 * does not fit the library's limits and the CTAs walk the unit order instead), or -1 for bad
 * arguments or units_cap below the unit count. Units are numbered in the kernel's unit order:
 * head blocks of head_block heads, inside a block the Q-tile pairs from the last one down, the
 * heads of the block next to each other. The caller owns every buffer. */
int attn_debug_schedule(int BH, int N_q, int N_k, int d, int G, int causal, int sms, int *units,
                        int units_cap, int *off, int *n_units, int *head_block);

/*
 * Cross-attention and grouped-query attention (the "natural extensions" named in the
 * "cuda-reranker" README): the forward of attn_fwd_path with separate query and key/value
 * shapes.
 *   q, o         fp16 [B, H, N_q, d]; lse (optional) fp32 [B, H, N_q]
 *   k, v         fp16 [B, H_kv, N_k, d]; H must be a multiple of H_kv. Query head h reads
 *                key/value head h / (H / H_kv) (groups of consecutive query heads share one
 *                K, V; H_kv = H is multi-head attention, H_kv = 1 multi-query attention)
 *   key_lengths  device int32 [B] or NULL: keys j >= key_lengths[b] (clamped to [0, N_k]) are
 *                excluded
 *   causal       query i sees keys j <= i + N_k - N_q: the diagonal is aligned at the last rows,
 *                so the last query sees every key (a query block appended to a sequence of
 *                N_k - N_q earlier tokens). The pages fix no alignment for N_q != N_k; this is
 *                the reading taken. Rows with no allowed key get O = 0 and lse = -inf.
 *   dtype        attn_dtype_t of q, k, v and o (all four the same): ATTN_DTYPE_F16, or
 *                ATTN_DTYPE_BF16 (tcgen05 kernel only), or ATTN_DTYPE_F32 (d = 32 only; see
 *                attn_dtype_t for its two paths); another value or d is ATTN_ERR_UNSUPPORTED
 *   path         ATTN_PATH_AUTO (the decoding kernel for fp16 and bf16 problems of at most
 *                16 query rows per head after packing over at least ATTN_DECODE_MIN_KEYS keys;
 *                else for fp16 self-attention shapes the kernel attn_auto_path selects, the
 *                fp32-accurate kernel for fp32, the tcgen05 kernel otherwise),
 *                ATTN_PATH_TCGEN05 or ATTN_PATH_WARP_MMA (fp16 and fp32); ATTN_PATH_SHORT
 *                takes fp16 self-attention shapes only (H_kv = H, N_q = N_k); ATTN_PATH_DECODE
 *                fp16 and bf16 with at most 16 query rows per head after packing; any other
 *                combination is ATTN_ERR_UNSUPPORTED.
 * B, H, H_kv, N_q, N_k >= 1 (else ATTN_ERR_INVALID_ARG, as is H not a multiple of H_kv); the
 * element count of every tensor must fit int64 and B*H int32. The other arguments, layouts
 * and errors are those of attn_fwd_lse. With H_kv = H, N_q = N_k and fp16 it is attn_fwd_path.
 * With H_kv < H and N_q < 128 the G = H / H_kv query heads of a group run as one problem of
 * G * N_q query rows (they are adjacent in q, o and lse), so they share Q tiles; under the causal
 * mask each packed row keeps its own query's diagonal. The result is the same.
 */
attn_status_t attn_fwd_ex(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                          int H, int H_kv, int N_q, int N_k, int d, int dtype, float sm_scale,
                          int causal, const int32_t *key_lengths, int path, attn_stream_t stream);

/*
 * Split-KV forward: the same result as attn_fwd_lse (lse may be NULL), computed with the keys
 * of every (batch*head, pair of 128-row query tiles) divided into n_splits contiguous ranges of
 * 128-key tiles that run as separate work units (more parallel work when B*H*ceil(N/256) is
 * below the SM count, e.g. one long sequence), followed by a merge of the ranges. The merge is
 * the combination of two partial softmaxes of "Self-Attention Kernel & Inference Engine from
 * Scratch" ("Online Softmax Formulation") applied to n_splits ranges at once: with lse_s the
 * logsumexp of range s and O_s its normalised output, lse = log sum_s exp(lse_s) and
 * O = sum_s exp(lse_s - lse) O_s.
 * Where every pair has the same number of key tiles (no causal mask, or N <= 256) and it
 * finishes sooner, the ranges are not equal parts of each pair: the key tiles of all pairs are
 * laid end to end and cut into one equal run per SM, and range s of a pair is its part of the
 * s-th run that touches it (a pair then has at most n_splits ranges, some possibly empty). The
 * result is the same attention either way.
 *   n_splits         1..16, or <= 0 for attn_splitkv_auto_splits(B, H, N, d, causal)
 *   workspace        device memory of at least attn_splitkv_workspace_bytes(B, H, N, d, n_splits)
 *                    bytes, 16-byte aligned, owned by the caller; its contents on entry do not
 *                    matter and on return are undefined. Launches that share a workspace must
 *                    not overlap on the device.
 * The other arguments, layouts and errors are those of attn_fwd_lse; a missing or too small
 * workspace or n_splits > 16 gives ATTN_ERR_INVALID_ARG, a misaligned one ATTN_ERR_MISALIGNED.
 * Runs the tcgen05 kernel (every d in {32, 64, 128}, every N) and one merge kernel.
 */
attn_status_t attn_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                               int B, int H, int N, int d, float sm_scale, int causal,
                               const int32_t *key_lengths, int n_splits, void *workspace,
                               size_t workspace_bytes, attn_stream_t stream);

/* Workspace bytes attn_fwd_splitkv needs: n_splits * B*H*N * (d + 1) * 4 (fp32 partial
 * outputs and logsumexps of every range). 0 for invalid sizes or n_splits outside 1..16. */
size_t attn_splitkv_workspace_bytes(int B, int H, int N, int d, int n_splits);

/* The split count attn_fwd_splitkv uses for n_splits <= 0, for the current device's SM count
 * (152, GB300's, where no device answers):
 * where every pair has the same key tile count and runs of equal length over all pairs (see
 * attn_fwd_splitkv) finish sooner than any equal split, the most runs that touch one pair;
 * otherwise, without a causal mask the most ranges that still give one (Q tile pair, key range) unit per
 * SM (SMs / pairs, rounded down); with it enough units that the largest is no longer than an
 * SM's average share (the largest pair's K/V tile count over the mean, about two, times SMs /
 * pairs, rounded up). At most one range per two 128-key tiles and at most 16; at least 1. -1
 * for invalid sizes. */
int attn_splitkv_auto_splits(int B, int H, int N, int d, int causal);

/* Split-KV forward of cross-attention and grouped-query attention: the result of attn_fwd_ex
 * (shapes, head groups, causal alignment and dtype as there), computed as attn_fwd_splitkv
 * computes it.
 * The workspace is sized by attn_splitkv_workspace_bytes(B, H, N_q, d, n_splits) (query rows);
 * n_splits <= 0 takes attn_splitkv_auto_splits_ex(B, H, H_kv, N_q, N_k, d, causal). With H_kv = H and
 * N_q = N_k and fp16 it is attn_fwd_splitkv. */
attn_status_t attn_fwd_splitkv_ex(const void *q, const void *k, const void *v, void *o, float *lse,
                                  int B, int H, int H_kv, int N_q, int N_k, int d, int dtype,
                                  float sm_scale, int causal, const int32_t *key_lengths,
                                  int n_splits, void *workspace, size_t workspace_bytes,
                                  attn_stream_t stream);

/*
 * Naive three-pass forward: the same attention as attn_fwd_lse, computed the textbook way with
 * the N x N score and probability matrices written to and read back from device memory ("Naive
 * Attention Kernel", sections "1. Standard Attention: Step by Step", "2. HBM Traffic Analysis"
 * and "3. Naive CUDA Implementation"; "Tensor Parallelism with CUDA - Standard Attention",
 * section "The Naive HBM Algorithm"). It is the library's comparison baseline for the traffic
 * the fused kernels avoid, not a path for production use:
 *   pass 1  S = sm_scale * Q K^T for every query/key pair of every head   (fp32, into workspace)
 *   pass 2  P = softmax(S + mask) row by row, and lse                     (fp16, into workspace)
 *   pass 3  O = P V over every key column of P                            (fp16, into o)
 * Scores excluded by the causal mask or the key lengths are computed and stored like the
 * others; the softmax pass gives them probability 0.
 *   workspace        device memory of at least attn_naive_workspace_bytes(B, H, N) bytes,
 *                    16-byte aligned, owned by the caller: S as fp32 [B*H, N, Np], then P as
 *                    fp16 [B*H, N, Np], with Np = N rounded up to a multiple of 128 (the padded
 *                    columns of P hold zeros). On return it holds S and P of this call. Launches
 *                    that share a workspace must not overlap on the device.
 * fp16 self-attention only ([B, H, N, d], d in {32, 64, 128}); the other arguments, layouts and
 * errors are those of attn_fwd_lse. A missing or too small workspace gives ATTN_ERR_INVALID_ARG,
 * a misaligned one ATTN_ERR_MISALIGNED. Three kernel launches on `stream`.
 */
attn_status_t attn_fwd_naive(const void *q, const void *k, const void *v, void *o, float *lse,
                             int B, int H, int N, int d, float sm_scale, int causal,
                             const int32_t *key_lengths, void *workspace, size_t workspace_bytes,
                             attn_stream_t stream);

/* Workspace bytes attn_fwd_naive needs: B*H*N*Np*6 (fp32 S and fp16 P, Np = N rounded up to a
 * multiple of 128); 0 for invalid sizes or a count that does not fit size_t. */
size_t attn_naive_workspace_bytes(int B, int H, int N);

/* attn_splitkv_auto_splits for the shapes of attn_fwd_ex (H query heads over H_kv key/value heads,
 * N_q query rows over N_k keys), counted on the problem the kernels run (query heads of a group
 * packed together where attn_fwd_ex packs them); under the causal mask the largest pair's work
 * over the mean is taken from the pairs' 128-key tile counts with the diagonal of attn_fwd_ex.
 * -1 for invalid sizes. */
int attn_splitkv_auto_splits_ex(int B, int H, int H_kv, int N_q, int N_k, int d, int causal);

/*
 * Split-KV forward that allocates nothing (the pages have no counterpart: this is a service of
 * the library). For callers that cannot allocate device memory where they call the attention:
 * a serving process whose device memory already belongs to its own pool or caching allocator,
 * a plug-in hosted by a runtime that gives it no allocator, or a latency-bound loop that cannot
 * pay the synchronisation of cudaMalloc/cudaFree. It is attn_fwd_splitkv with its workspace
 * in a fixed array of attn_noalloc_scratch_bytes() bytes (64 MiB) that is part of the
 * library's device code: every GPU on which the library is loaded holds that array until the
 * process exits. The caller passes inputs and outputs only; no call allocates, in this
 * library or in any library it calls.
 *   - n_splits <= 0 takes the automatic count (attn_splitkv_auto_splits), lowered to the
 *     largest count whose workspace fits the array.
 *   - A problem whose split-KV workspace (attn_splitkv_workspace_bytes) exceeds the array
 *     (for the automatic count: even with one range) returns ATTN_ERR_SCRATCH_LIMIT before
 *     any launch; use fewer splits or attn_fwd_splitkv.
 *   - The array belongs to the library's device code. The CUDA driver reserves it on a GPU
 *     when it loads that code there, which with lazy module loading (the default) happens at
 *     the first call of this entry point on the device, not when the library is opened. The
 *     same first call looks up the array's device address (once per device, with that device
 *     current). A caller that must not see any reservation on its hot path makes one warm-up
 *     call on each device first, outside any stream capture.
 *   - Every call on a device shares the one array, which keeps the last call's contents (no
 *     part of it needs clearing: each call writes all it reads). Calls whose executions overlap
 *     on the same GPU (different streams, concurrent host threads) race on it and must be
 *     ordered by the caller.
 * Arguments and the other errors are those of attn_fwd_splitkv without the workspace.
 */
attn_status_t attn_fwd_splitkv_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                                       int B, int H, int N, int d, float sm_scale, int causal,
                                       const int32_t *key_lengths, int n_splits, attn_stream_t stream);

/* Bytes of the fixed scratch array of attn_fwd_splitkv_noalloc (64 MiB). */
size_t attn_noalloc_scratch_bytes(void);

/* The kernel ATTN_PATH_AUTO selects for sequence length N and head dimension d
 * (an attn_path_t value), or -1 when d is unsupported. No CUDA call is made. */
int attn_auto_path(int N, int d);

/* The kernel ATTN_PATH_AUTO selects in attn_fwd_ex for H query heads over H_kv key/value heads,
 * N_q query rows over N_k keys, head dimension d, element type dtype (attn_dtype_t) and the
 * causal flag (an attn_path_t value), or -1 for invalid or unsupported arguments. The batch
 * size and key lengths do not enter the choice. No CUDA call is made. */
int attn_auto_path_ex(int H, int H_kv, int N_q, int N_k, int d, int dtype, int causal);

/* Static description of a status code. Never NULL. */
const char *attn_status_str(attn_status_t status);

/* Synchronizes `stream`, then reads and clears the device-side status word of
 * the current device: ATTN_OK, or ATTN_ERR_TIMEOUT when a bounded wait in an
 * earlier launch ran out. ATTN_ERR_CUDA if the synchronization fails. */
attn_status_t attn_read_device_status(attn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_ATTN_H */
