/*
 * vlf.h -- C ABI of libvlf.so: fused variable-length flash attention (forward and backward)
 * for NVIDIA GB300 (sm_103a).
 *
 * The operation is the one the mtlattn 0.3.0 page defines for its varlen_attention call
 * (section "Use"):
 *   q [total_q, H_q, D_qk], k [total_kv, H_kv, D_qk], v [total_kv, H_kv, D_v], packed by
 *   cumulative sequence lengths cu_seqlens_q / cu_seqlens_kv (int32 [num_seqs + 1]), no padding;
 *   query head h reads kv head h / (H_q / H_kv) (GQA / MQA);
 *   logit(i, j) = scale * (q_i . k_j) + bias[global row i, h or 0, sequence-local key j];
 *   causal (end-aligned): row i sees key j iff j <= i + (kv_len - q_len);
 *   window W > 0: row i sees only the last W keys up to that diagonal,
 *                 j >= i + (kv_len - q_len) - W + 1;
 *   out_i = softmax_j(logit(i, .)) v, accumulated in fp32 without materialising the L x L
 *   score matrix (online softmax, mtlattn 0.3.0 header; triton-msl part 1, "What works").
 * The asymmetric latent-attention head (D_qk = 192 = 128 "nope" ++ 64 "rope", D_v = 128) is the
 * one of triton-msl part 2, "Latent attention".
 *
 * Conventions for every entry point
 *   - All tensors are dense, row-major (C-contiguous) device buffers owned by the caller; the
 *     library never allocates, frees or synchronises inside vlf_attn_varlen_fwd/_bwd and only
 *     enqueues work on `stream` (mtlattn 0.3.0, "Notes": work is ordered on the caller's stream
 *     without a per-call host sync).
 *   - Element types: q, k, v, out, dout, dq, dk, dv share `dtype` (VLF_F16, VLF_BF16, VLF_F32);
 *     bias, lse and the workspace are fp32.  Accumulation is fp32 for every dtype; each output is
 *     rounded once (round-to-nearest-even) to its storage type.
 *   - Every pointer must be 16-byte aligned.
 *   - Correct-or-refuse (triton-msl part 1, "Correct-or-refuse"): an argument the library cannot
 *     handle returns a negative vlf_status before anything is enqueued; nothing is silently
 *     approximated.  Errors found on the device (bad cu_seqlens, a pipeline wait that ran out of
 *     time) are recorded in a per-device error word and returned by vlf_check_error().  The
 *     kernels never trap.
 *   - Indices into q/k/v/out/bias are 64-bit: bias tensors beyond 2^32 elements are supported.
 */
#ifndef VLF_H
#define VLF_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st *vlf_stream_t;

typedef enum { VLF_F16 = 0, VLF_BF16 = 1, VLF_F32 = 2 } vlf_dtype;

typedef enum {
  VLF_OK = 0,
  VLF_ERR_INVALID = -1,     /* null pointer, negative size, H_q % H_kv != 0, bias_heads not 1/H_q */
  VLF_ERR_UNSUPPORTED = -2, /* a valid problem this build does not implement (e.g. head width) */
  VLF_ERR_ALIGN = -3,       /* a pointer is not 16-byte aligned (device: a kernel's shared window
                               is not 1024-byte aligned) */
  VLF_ERR_LAUNCH = -4,      /* the CUDA runtime refused a launch or a query */
  VLF_ERR_TIMEOUT = -5,     /* device: a pipeline wait exceeded its time limit (kernel bailed out) */
  VLF_ERR_BAD_SEQLENS = -6, /* device: cu_seqlens not in [0, total], decreasing, or longer than max_seqlen */
  VLF_ERR_WORKSPACE = -7    /* a workspace missing or smaller than its size query returns */
} vlf_status;

/* Extended-call flags (vlf_attn_varlen_fwd_ex / _bwd_ex). */
#define VLF_FLAG_NO_SKIP 1u    /* visit every KV tile, masking per element (tile-skip check) */
#define VLF_FLAG_FORCE_SIMT 2u /* use the SIMT fp32-FMA kernels even where a tensor-core one exists */
#define VLF_FLAG_NO_PACK 4u    /* forward: never pack a kv head's query heads into one tile (the
                                  decode-size layout); results are identical either way */
#define VLF_FLAG_TEST_TIMEOUT 8u /* testing the failure path: the tensor-core forward's producer
                                    never loads the query tile, so every CTA's pipeline waits run
                                    out after their time limit (2 s); the kernel records
                                    VLF_ERR_TIMEOUT, drains, frees its TMEM and returns, and the
                                    device stays usable (out is not written) */

/*
 * Forward.  mtlattn 0.3.0, section "Use" (varlen_attention with scale, causal, window, attn_bias).
 *
 *   q            [total_q, h_q, d_qk]      dtype
 *   k            [total_kv, h_kv, d_qk]    dtype
 *   v            [total_kv, h_kv, d_v]     dtype
 *   cu_seqlens_q / cu_seqlens_kv           device int32 [num_seqs + 1], cu[0] = 0,
 *                                          non-decreasing, cu[num_seqs] = total_q / total_kv
 *   max_seqlen_q / max_seqlen_kv           host ints >= every sequence's q_len / kv_len
 *                                          (size the launch grid; max_seqlen_kv is also the
 *                                          row length of `bias`)
 *   h_q % h_kv == 0
 *   scale        softmax scale; <= 0 selects 1/sqrt(d_qk)
 *   causal       0/1, end-aligned
 *   window       <= 0: none; else the number of keys each row sees up to its diagonal
 *   bias         NULL or fp32 [total_q, bias_heads, max_seqlen_kv], bias_heads in {1, h_q};
 *                row = global query row, column = sequence-local key; -inf masks the pair
 *   out          [total_q, h_q, d_v]       dtype (written)
 *   lse          NULL or fp32 [h_q, total_q]: natural-log log-sum-exp of each row's logits,
 *                -inf for a row that sees no key (its out row is 0).  Required by the backward.
 * Supported: dtype F16/BF16 with any 1 <= d_qk, d_v <= 256 (tensor-core kernels for
 * (d_qk, d_v) in {(64,64), (96,96), (128,128), (192,128), (256,256)}); dtype F32 with d_qk,
 * d_v <= 256 (tensor-core kernels for (32,32) and (64,64), products in three tf32 passes with
 * fp32 accumulation; fp32 FMA otherwise).
 */
int vlf_attn_varlen_fwd(const void *q, const void *k, const void *v,
                        const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_kv, int num_seqs,
                        int total_q, int total_kv, int max_seqlen_q, int max_seqlen_kv,
                        int h_q, int h_kv, int d_qk, int d_v, int dtype,
                        float scale, int causal, int window,
                        const float *bias, int bias_heads,
                        void *out, float *lse, vlf_stream_t stream);

/*
 * As vlf_attn_varlen_fwd, plus `flags` (VLF_FLAG_*) and `bias_bands`: NULL, or the result of
 * vlf_bias_bands for this bias (below), which lets the kernels skip the KV tiles the bias masks
 * for every row of a query tile.
 */
int vlf_attn_varlen_fwd_ex(const void *q, const void *k, const void *v,
                           const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_kv, int num_seqs,
                           int total_q, int total_kv, int max_seqlen_q, int max_seqlen_kv,
                           int h_q, int h_kv, int d_qk, int d_v, int dtype,
                           float scale, int causal, int window,
                           const float *bias, int bias_heads,
                           void *out, float *lse, vlf_stream_t stream, unsigned flags,
                           const void *bias_bands);

/*
 * Split-KV forward, for problems whose (query tile, head) CTAs are too few to fill the GPU --
 * small batches of decode steps (one query row per sequence against a long cache; the
 * end-aligned causal rule serves cached decode, mtlattn 0.3.0, "Use") or short queries against
 * long keys.
 * Each CTA's KV band is cut into num_splits contiguous parts computed in parallel; each part
 * writes its normalised fp32 result and its log-sum-exp L_s to the workspace, and a combine
 * kernel writes out = sum_s exp(L_s - LSE) out_s and lse = LSE = log sum_s exp(L_s) -- the
 * same softmax, summed in another order (results agree with vlf_attn_varlen_fwd to rounding).
 *
 *   arguments as vlf_attn_varlen_fwd_ex, plus
 *   num_splits   0: the library's choice (vlf_fwd_num_splits); 1: unsplit; 2..64: that many
 *                parts (some may be empty); num_splits * num_seqs <= 65535
 *   workspace    device buffer of at least vlf_attn_varlen_fwd_split_workspace_size(total_q,
 *                h_q, d_v, num_splits) bytes, owned by the caller, clobbered; may be NULL when
 *                the call runs unsplit
 * Shapes that cannot split (dtype F32, (d_qk, d_v) other than (64,64), (96,96), (128,128),
 * (256,256)) run the unsplit forward.  Returns VLF_ERR_WORKSPACE when a split call's workspace is missing or
 * too small.
 */
int vlf_attn_varlen_fwd_split(const void *q, const void *k, const void *v,
                              const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_kv,
                              int num_seqs, int total_q, int total_kv, int max_seqlen_q,
                              int max_seqlen_kv, int h_q, int h_kv, int d_qk, int d_v, int dtype,
                              float scale, int causal, int window,
                              const float *bias, int bias_heads,
                              void *out, float *lse, int num_splits,
                              void *workspace, size_t workspace_bytes, vlf_stream_t stream,
                              unsigned flags, const void *bias_bands);

/*
 * The number of parts vlf_attn_varlen_fwd_split uses for num_splits = 0 (1: no split).  Pure
 * host arithmetic on the launch shape, with the CTAs resident per SM (two; one at width 256)
 * as the "slots" of a wave:
 * a grid below one wave is split into as many parts as keep it within one wave, each part at
 * least 256 keys (at most 64 parts); a grid of one to three waves whose last wave is under 95%
 * full gets 2 or 3 parts, whichever fills its waves better (the fewer on a tie), each at least
 * 1024 keys; larger grids are not split.  num_sms <= 0 takes the current device's SM count
 * (returns 1 if it cannot be queried).
 */
int vlf_fwd_num_splits(int num_seqs, int max_seqlen_q, int max_seqlen_kv, int h_q, int h_kv,
                       int d_qk, int d_v, int dtype, unsigned flags, int num_sms);

/*
 * Bytes of workspace vlf_attn_varlen_fwd_split needs: fp32 parts [num_splits, total_q, h_q, d_v]
 * and their log-sum-exps [num_splits, h_q, total_q], each rounded up to 256 bytes; 0 when
 * num_splits < 2.  Pure host arithmetic.
 */
size_t vlf_attn_varlen_fwd_split_workspace_size(int total_q, int h_q, int d_v, int num_splits);

/*
 * Bytes of fp32 workspace vlf_attn_varlen_bwd needs: the row dot products D = rowsum(dO o O),
 * [h_q, total_q] fp32 (rounded up to 256 bytes).  Pure host arithmetic; never fails (returns 0
 * for invalid sizes).
 */
size_t vlf_attn_varlen_bwd_workspace_size(int total_q, int total_kv, int h_q, int h_kv,
                                          int d_qk, int d_v, int dtype);

/*
 * Backward.  The gradients of sum(out * dout) with respect to q, k, v, the bias held constant
 * (mtlattn 0.3.0, "Use": the bias is treated as constant; triton-msl part 2, "Beyond softmax":
 * a tiled FlashAttention-2 backward).  Same shapes and conventions as the forward, plus
 *   out, lse     the forward's outputs for the same inputs
 *   dout         [total_q, h_q, d_v]       dtype
 *   dq           [total_q, h_q, d_qk]      dtype (written)
 *   dk, dv       [total_kv, h_kv, d_qk], [total_kv, h_kv, d_v] dtype (written; each kv head
 *                sums the contributions of its h_q / h_kv query heads)
 *   workspace    device buffer of at least vlf_attn_varlen_bwd_workspace_size(...) bytes,
 *                owned by the caller, contents need not be initialised; clobbered.
 */
int vlf_attn_varlen_bwd(const void *q, const void *k, const void *v, const void *out,
                        const float *lse, const void *dout,
                        const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_kv, int num_seqs,
                        int total_q, int total_kv, int max_seqlen_q, int max_seqlen_kv,
                        int h_q, int h_kv, int d_qk, int d_v, int dtype,
                        float scale, int causal, int window,
                        const float *bias, int bias_heads,
                        void *dq, void *dk, void *dv,
                        void *workspace, size_t workspace_bytes, vlf_stream_t stream);

/*
 * As vlf_attn_varlen_bwd, plus `flags`, optional per-stage timing events and the bias bands
 * (NULL, or vlf_bias_bands's result for this bias, as in vlf_attn_varlen_fwd_ex).  When
 * stage_events is not NULL it holds n_stage_events >= VLF_BWD_STAGES + 1 cudaEvent_t handles
 * (created by the caller); event 0 is recorded on `stream` before the first kernel and event
 * s+1 after stage s, stages being, in order: 0 the dO.O row-dot pre-pass, 1 the dK/dV kernel,
 * 2 the dQ kernel.  Recording adds no synchronisation.
 */
#define VLF_BWD_STAGES 3
int vlf_attn_varlen_bwd_ex(const void *q, const void *k, const void *v, const void *out,
                           const float *lse, const void *dout,
                           const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_kv, int num_seqs,
                           int total_q, int total_kv, int max_seqlen_q, int max_seqlen_kv,
                           int h_q, int h_kv, int d_qk, int d_v, int dtype,
                           float scale, int causal, int window,
                           const float *bias, int bias_heads,
                           void *dq, void *dk, void *dv,
                           void *workspace, size_t workspace_bytes, vlf_stream_t stream,
                           unsigned flags, void *const *stage_events, int n_stage_events,
                           const void *bias_bands);

/*
 * Bias bands.  An additive bias often masks whole stretches of each row (mtlattn 0.3.0, "Use":
 * -inf masks a pair and a boolean mask becomes a 0 / -inf bias; a prefix-LM mask hides every key
 * past the prefix and the diagonal).  This pass records, for each bias head and query row, the
 * keys from the first to the last finite value among the row's first kv_len columns, and whether
 * the bias is exactly 0 throughout them; and the same, combined, for each block of 64 rows of
 * each sequence.  Given to the _ex calls, it lets the tensor-core kernels (16-bit data, widths
 * up to 128, one query tile per CTA) skip the KV tiles and query items that hold only -inf bias
 * values for their rows -- the skipped pairs contribute exact zeros -- and mask by interval
 * without reading the bias where every row of a tile is such a 0 / -inf interval.  The results
 * equal those computed without the bands within the stated tolerances (the bias values of a pure
 * interval are 0; the masked pairs are the same).  The bands must come from this bias (same
 * tensor, unmodified since): stale bands give wrong results.
 *   bias, bias_heads, cu_seqlens_q / _kv, num_seqs, total_q, max_seqlen_kv   as in the forward
 *   bands        device buffer of at least vlf_bias_bands_size(total_q, bias_heads) bytes,
 *                16-byte aligned, owned by the caller, written: two int32x4 tables of
 *                [bias_heads][total_q] entries -- per row {lo, hi, pure, 0} (keys [lo, hi) from
 *                the first to the last finite value, lo = hi = 0 if none; pure 1 when the bias
 *                is 0 throughout them), then per 64-row block of each sequence, at the block's
 *                first row, {lo, hi, ilo, ihi}: the union of its rows' intervals and, when all
 *                its rows are pure, their intersection (-1, -1 otherwise)
 * Enqueued on `stream`; no synchronisation.  Returns VLF_OK or a negative status (invalid
 * arguments, VLF_ERR_WORKSPACE for a missing or short buffer).
 */
size_t vlf_bias_bands_size(int total_q, int bias_heads);
int vlf_bias_bands(const float *bias, int bias_heads, const int32_t *cu_seqlens_q,
                   const int32_t *cu_seqlens_kv, int num_seqs, int total_q, int max_seqlen_kv,
                   void *bands, size_t bands_bytes, vlf_stream_t stream);

/*
 * Latent attention with split operands (triton-msl part 2, "Latent attention": the score is the
 * sum of two query-key products over different widths, a 128-wide "nope" part and a 64-wide
 * "rope" part, so the contraction is 192 wide while the output stays 128 wide).  The parts are
 * passed as they are produced, without concatenation, and the rope key may be one tensor shared
 * by every head:
 *   logit(i, j) = scale * (q_nope_i . k_nope_j + q_rope_i . k_rope_j) + bias,
 * with head h reading k_nope / v of kv head h / (h_q / h_kv) and k_rope of that kv head, or of
 * the single rope head when rope_heads = 1.  Results equal vlf_attn_varlen_fwd / _bwd on the
 * concatenated operands q = [q_nope | q_rope], k = [k_nope | k_rope broadcast over kv heads]
 * (the same kernels, the same arithmetic).
 *
 *   q_nope  [total_q, h_q, 128]   q_rope [total_q, h_q, 64]          dtype
 *   k_nope  [total_kv, h_kv, 128] k_rope [total_kv, rope_heads, 64]  dtype, rope_heads in {1, h_kv}
 *   v       [total_kv, h_kv, 128]                                     dtype
 *   d_nope, d_rope, d_v must be 128, 64, 128 (VLF_ERR_UNSUPPORTED otherwise, and for dtype F32
 *   or VLF_FLAG_FORCE_SIMT: there is no SIMT kernel for split operands); other arguments and
 *   outputs as vlf_attn_varlen_fwd / _bwd.  scale <= 0 selects 1/sqrt(192).
 * Backward outputs (written): dq_nope / dq_rope like q_nope / q_rope, dk_nope like k_nope, dv
 * like v, dk_rope like k_rope -- for a shared rope key (rope_heads = 1) the sum over every head
 * of its gradient, accumulated in fp32 in kv-head order (deterministic) and rounded once.  The
 * workspace (caller-owned, clobbered) holds the row dot products and, for a shared rope key with
 * h_kv > 1, the per-kv-head fp32 rope gradients [h_kv, total_kv, 64].
 */
int vlf_attn_varlen_fwd_latent(const void *q_nope, const void *q_rope, const void *k_nope,
                               const void *k_rope, const void *v,
                               const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_kv,
                               int num_seqs, int total_q, int total_kv, int max_seqlen_q,
                               int max_seqlen_kv, int h_q, int h_kv, int rope_heads,
                               int d_nope, int d_rope, int d_v, int dtype,
                               float scale, int causal, int window,
                               const float *bias, int bias_heads,
                               void *out, float *lse, vlf_stream_t stream, unsigned flags);

/* Bytes of workspace vlf_attn_varlen_bwd_latent needs (pure host arithmetic; 0 for invalid
 * sizes). */
size_t vlf_attn_varlen_bwd_latent_workspace_size(int total_q, int total_kv, int h_q, int h_kv,
                                                 int rope_heads, int dtype);

int vlf_attn_varlen_bwd_latent(const void *q_nope, const void *q_rope, const void *k_nope,
                               const void *k_rope, const void *v, const void *out,
                               const float *lse, const void *dout,
                               const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_kv,
                               int num_seqs, int total_q, int total_kv, int max_seqlen_q,
                               int max_seqlen_kv, int h_q, int h_kv, int rope_heads,
                               int d_nope, int d_rope, int d_v, int dtype,
                               float scale, int causal, int window,
                               const float *bias, int bias_heads,
                               void *dq_nope, void *dq_rope, void *dk_nope, void *dk_rope,
                               void *dv, void *workspace, size_t workspace_bytes,
                               vlf_stream_t stream, unsigned flags,
                               void *const *stage_events, int n_stage_events);

/*
 * Number of kernels this library has launched in this process (all devices, all streams),
 * counted on the host at each successful launch.  For benchmarks that report their launches.
 */
uint64_t vlf_launch_count(void);

/*
 * Which kernel family the forward / backward would use for this problem: 1 tensor-core
 * (tcgen05), 0 SIMT fp32 FMA, negative status if the problem is refused.  Host only.
 */
int vlf_fwd_path(int h_q, int h_kv, int d_qk, int d_v, int dtype, int bias_heads, unsigned flags);
int vlf_bwd_path(int h_q, int h_kv, int d_qk, int d_v, int dtype, int bias_heads, unsigned flags);

/*
 * Synchronises `stream`, then returns and clears the current device's error word (VLF_OK,
 * VLF_ERR_TIMEOUT or VLF_ERR_BAD_SEQLENS), or VLF_ERR_LAUNCH if the CUDA runtime reports an
 * error.  The only entry point that blocks the host.
 */
int vlf_check_error(vlf_stream_t stream);

/* Static description of a status code. */
const char *vlf_status_string(int status);

/*
 * Tile scheduler (host-callable, no GPU needed).  For sequence-local query rows [r0, r1) of a
 * sequence with q_len queries and kv_len keys, the key range [*lo, *hi) that holds every key
 * any of those rows may see under the causal/window rules above; keys outside it are skipped
 * whole (mtlattn 0.3.0, "Use": fully masked KV tiles are skipped, window jumps to its band).
 * Returns VLF_OK or VLF_ERR_INVALID.
 */
int vlf_sched_kv_band(int r0, int r1, int q_len, int kv_len, int causal, int window,
                      int *lo, int *hi);

/* The query rows [*lo, *hi) that may see any key of [j0, j1) (the backward's dK/dV band). */
int vlf_sched_q_band(int j0, int j1, int q_len, int kv_len, int causal, int window,
                     int *lo, int *hi);

/*
 * Backward that allocates nothing.  The pages have no counterpart to this entry point; it exists
 * for callers that cannot allocate device memory at call time -- a plugin whose enqueue hook may
 * not allocate, a service that reserves its memory budget up front, or code that must not
 * trigger the device-wide synchronisation cudaMalloc / cudaFree can cause.  Same arguments and
 * results as vlf_attn_varlen_bwd without the workspace: the row dot products live in a
 * fixed-size array inside the library's own device memory instead.
 *   - Size limit: h_q * total_q <= 8,388,608 (vlf_noalloc_scratch_bytes() bytes of fp32);
 *     larger problems return VLF_ERR_UNSUPPORTED before anything is enqueued.
 *   - Every GPU that loads the library holds that array (32 MiB) until the process exits.
 *   - Calls on one device share the array and it keeps the last call's contents (nothing in it
 *     needs to start at zero).  Calls whose work overlaps on the GPU race on it: order them on
 *     one stream, or with events.
 *   - The first call on each device looks up the array's device address; make that first call
 *     before any stream capture begins.  The address is kept for the life of the process and is
 *     not valid after a cudaDeviceReset of that device: do not call this entry point on a
 *     device after resetting it.
 *   - No cudaMalloc, cudaFree or other allocating routine is called.
 */
int vlf_attn_varlen_bwd_noalloc(const void *q, const void *k, const void *v, const void *out,
                                const float *lse, const void *dout,
                                const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_kv,
                                int num_seqs, int total_q, int total_kv, int max_seqlen_q,
                                int max_seqlen_kv, int h_q, int h_kv, int d_qk, int d_v, int dtype,
                                float scale, int causal, int window,
                                const float *bias, int bias_heads,
                                void *dq, void *dk, void *dv, vlf_stream_t stream);

/* Bytes of the fixed array vlf_attn_varlen_bwd_noalloc uses as its workspace. */
size_t vlf_noalloc_scratch_bytes(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int vlf_version(void);

#ifdef __cplusplus
}
#endif

#endif /* VLF_H */
