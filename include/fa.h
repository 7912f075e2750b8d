/*
 * fa.h - C ABI of the GB300 (sm_103a) fused exact-attention library, libfa.so.
 *
 * Computes O = softmax(scale * Q K^T [+ causal or 128x128 block mask]) V without writing the
 * N x N score or probability matrices to memory, plus its gradient.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  Layout    Q, K, V, O, dO, dQ, dK, dV are dense, contiguous [B, H, N, d] tensors of one
 *            16-bit type (FA_FP16 or FA_BF16) in device memory; row (b, h, n) starts at element
 *            ((b * H + h) * N + n) * d.  LSE and the backward scratch D are fp32 [B, H, N].
 *            Every device pointer must be 16-byte aligned.
 *  Sizes     d is 64 or 128 (anything else: FA_ERR_UNSUPPORTED).  N >= 1 (ragged N is fine),
 *            B >= 1, H >= 1, B * H * N < 2^31.  scale must be finite and > 0.
 *  Masks     causal != 0: query i sees keys j <= i (queries and keys share one index).
 *            block_mask: device uint8 [T][T] row-major with T = ceil(N / 128), shared by every
 *            (b, h); entry (i, j) != 0 keeps the 128 x 128 score block of query rows
 *            [128 i, 128 i + 128) and key rows [128 j, 128 j + 128).  With both, a score is kept
 *            only if both keep it.  A query row whose every key is masked gets O = 0,
 *            LSE = -inf and zero gradients.  With a block mask T may not exceed 46340
 *            (N <= 5931520; T x T stays below 2^31), else FA_ERR_INVALID.
 *  Ownership The caller owns every buffer.  The library allocates no device memory on any
 *            call; it keeps one device status word per device, created on first use.
 *  Streams   Every call only enqueues work on `stream` (a cudaStream_t; NULL = legacy default
 *            stream) and returns.  The return code covers argument validation and launch
 *            errors only.  Device-side failures (a pipeline wait that ran out of time) are
 *            recorded in the status word and reported by fa_sync_status().
 *  Errors    0 on success, a negative FA_ERR_* code otherwise; nothing is launched when
 *            validation fails.  fa_status_string() names a code.
 *
 * The operation is the one defined by the pages this library follows:
 *  - "FlashAttention-2: better parallelism and work partitioning" (reading notes,
 *    zhongzhuzhou.org): standard attention eq. (2)-(4); forward Algorithm 1 with delayed
 *    normalisation eq. (10)-(11) and the logsumexp eq. (15); backward Algorithm 2 with
 *    P = exp(S - L) eq. (16) and the softmax Jacobian eq. (17); causal masking section.
 *  - FlashAttention post (bluuewhale.github.io): the 1/sqrt(d) scale ("How Attention Is
 *    Computed") and block-sparse FlashAttention ("Block-Sparse FlashAttention").
 *  - The same reading notes, section on MQA/GQA support, for the *_gqa entry points.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { FA_FP16 = 0, FA_BF16 = 1 } fa_dtype;

enum {
    FA_OK = 0,
    FA_ERR_INVALID = -1,      /* null or misaligned pointer, bad size, bad scale */
    FA_ERR_UNSUPPORTED = -2,  /* head dimension other than 64/128, or no sm_103 device */
    FA_ERR_CUDA = -3,         /* a CUDA runtime call failed (launch, attribute, symbol) */
    FA_ERR_TIMEOUT = -4,      /* a device pipeline wait ran out of time (from fa_sync_status) */
    FA_ERR_INTERNAL = -5      /* a kernel found its shared memory misplaced (its base not
                                 1024-byte aligned) and returned without computing; never
                                 expected (from fa_sync_status) */
};

/*
 * Forward.  FlashAttention-2 reading notes, Algorithm 1 (forward) and eq. (15).
 *   q, k, v : [B,H,N,d] inputs (device).
 *   o       : [B,H,N,d] output (device), same dtype.
 *   lse     : [B,H,N] fp32 output (device): LSE_i = m_i + ln(l_i) of the scaled scores.
 *   scale   : multiplies Q K^T before the softmax (1/sqrt(d) for standard attention).
 */
int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int N,
           int d, int dtype, float scale, int causal, void *stream);

/*
 * Block-sparse forward.  FlashAttention post, "Block-Sparse FlashAttention": a 128 x 128 score
 * block whose mask entry is zero is skipped entirely (never loaded, never multiplied).
 *   block_mask : device uint8 [ceil(N/128)][ceil(N/128)], must not be NULL.
 * Other arguments as fa_fwd.
 */
int fa_fwd_blocksparse(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                       int H, int N, int d, int dtype, float scale, int causal,
                       const uint8_t *block_mask, void *stream);

/*
 * Grouped-query forward.  FlashAttention-2 reading notes, MQA/GQA section: K and V have H_kv
 * heads, H_kv divides H, and query head h attends with K/V head h / (H / H_kv) (consecutive
 * query heads share a K/V head; H_kv = 1 is MQA, H_kv = H is fa_fwd).  K/V are read in place,
 * never copied per query head.
 *   q, o       : [B,H,N,d];  k, v : [B,H_kv,N,d];  lse : [B,H,N] fp32.
 *   block_mask : NULL for dense, otherwise as in fa_fwd_blocksparse.
 * H_kv < 1, or H_kv not dividing H: FA_ERR_INVALID.  Other arguments as fa_fwd.
 */
int fa_fwd_gqa(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
               int H_kv, int N, int d, int dtype, float scale, int causal,
               const uint8_t *block_mask, void *stream);

/*
 * Forward on 8-bit float inputs.  The forward of fa_fwd_gqa with Q, K, V given as e4m3 codes
 * (OCP 8-bit float E4M3: bias 7, 3 mantissa bits, largest 448, NaN = 0x7F/0xFF) and one scale
 * per tensor: element x of Q stands for e4m3(x) * descale_q (likewise K, V).  QK^T and PV run
 * as e4m3 tensor-core products (twice the bf16 rate); the softmax is fp32 as in fa_fwd; the
 * probabilities are rounded to e4m3 before PV (their largest values scaled near the top of the
 * e4m3 range), which bounds O's accuracy by e4m3's 3-bit mantissa rather than bf16's 8 bits.
 *   q       : [B,H,N,d] e4m3 codes (device);  k, v : [B,H_kv,N,d] e4m3 codes (device).
 *   o       : [B,H,N,d] bf16 output (device);  lse : [B,H,N] fp32 output, as in fa_fwd.
 *   descale_q, descale_k, descale_v : finite, > 0.
 *   workspace : at least fa_fwd_fp8_workspace_bytes() bytes, 16-byte aligned: V transposed
 *               ([B,H_kv,d,N rounded up to 16]), written by this call.
 *   block_mask : NULL for dense, otherwise as in fa_fwd_blocksparse.
 * d is 64 or 128.  Other arguments and errors as fa_fwd_gqa.
 */
size_t fa_fwd_fp8_workspace_bytes(int B, int H_kv, int N, int d);
int fa_fwd_fp8(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
               int H_kv, int N, int d, float scale, float descale_q, float descale_k,
               float descale_v, int causal, const uint8_t *block_mask, void *workspace,
               size_t workspace_bytes, void *stream);

/* Bytes of device scratch fa_bwd needs: D (fp32 [B,H,N]), rounded up to 256 bytes. */
size_t fa_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * Backward.  FlashAttention-2 reading notes, Algorithm 2 with the atomic dQ update replaced by
 * a separate dQ pass: D = rowsum(dO o O) (fa_bwd_preprocess), then dK and dV per key tile
 * (fa_bwd_dkdv), then dQ per query tile (fa_bwd_dq).  Deterministic: no atomics.
 *   o, lse     : the forward's outputs for these q, k, v (same scale, causal, mask).
 *   dout       : [B,H,N,d] gradient of the loss with respect to O.
 *   dq, dk, dv : [B,H,N,d] outputs (device), same dtype as q.
 *   workspace  : device scratch of at least fa_bwd_workspace_bytes() bytes, 16-byte aligned;
 *                overwritten, needs no initialisation.
 *   block_mask : NULL for dense, otherwise as in fa_fwd_blocksparse.
 */
int fa_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
           const float *lse, void *dq, void *dk, void *dv, void *workspace,
           size_t workspace_bytes, int B, int H, int N, int d, int dtype, float scale,
           int causal, const uint8_t *block_mask, void *stream);

/*
 * Bytes of device scratch fa_bwd_gqa needs: D (fp32 [B,H,N], rounded up to 256 bytes) plus,
 * when the dK/dV pass splits each K/V head's query group over several CTAs (few K/V heads, so
 * that the GPU is still filled), fp32 partial sums of dK and dV: 2 * splits * B*H_kv*N*d floats.
 * Returns 0 for invalid sizes.  Depends only on the arguments (and fa_debug_set_dkdv_splits).
 */
size_t fa_bwd_gqa_workspace_bytes(int B, int H, int H_kv, int N, int d);

/*
 * Grouped-query backward.  FlashAttention-2 reading notes, MQA/GQA section: the gradient of a
 * shared K/V head is the sum of its query heads' gradients.  The dK/dV pass walks all query
 * heads of a group through one accumulator in tensor memory (and, when split, adds the fp32
 * partials in a fixed order), so the result is deterministic.
 *   q, o, dout, dq : [B,H,N,d];  k, v, dk, dv : [B,H_kv,N,d];  lse : [B,H,N] fp32.
 *   workspace      : at least fa_bwd_gqa_workspace_bytes() bytes, 16-byte aligned.
 * Other arguments as fa_bwd; fa_bwd is this call with H_kv = H.
 */
int fa_bwd_gqa(const void *q, const void *k, const void *v, const void *o, const void *dout,
               const float *lse, void *dq, void *dk, void *dv, void *workspace,
               size_t workspace_bytes, int B, int H, int H_kv, int N, int d, int dtype,
               float scale, int causal, const uint8_t *block_mask, void *stream);

/*
 * Dropout on the attention probabilities (FlashAttention paper detail: dropout is one of the
 * operations fused into the kernel, O = dropout(softmax(S)) V; the pages give no generator).
 * Score (q, k) of query head b*H + h is dropped with probability t / 256, t = the nearest
 * integer to 256 * p_drop (ties to even), and a kept probability is scaled by 256 / (256 - t).
 * The decision is byte (k mod 16) of Philox4x32-10 (Salmon et al., SC 2011) with counter
 * (k div 16, q, b*H + h, offset) and key (seed mod 2^32, seed div 2^32), kept when that byte is
 * >= t; the backward regenerates the same decisions from the same arguments, so nothing is
 * stored.  offset must be below 2^32 (otherwise FA_ERR_INVALID).
 * fa_fwd_dropout: as fa_fwd_gqa; LSE is that of the scores (dropout does not change it).
 * fa_bwd_dropout: as fa_bwd_gqa (same workspace) for the forward with these dropout arguments.
 *   p_drop : 0 <= p_drop < 1 with t <= 255 (otherwise FA_ERR_INVALID); t = 0 is no dropout.
 */
int fa_fwd_dropout(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                   int H, int H_kv, int N, int d, int dtype, float scale, int causal,
                   const uint8_t *block_mask, float p_drop, unsigned long long seed,
                   unsigned long long offset, void *stream);
int fa_bwd_dropout(const void *q, const void *k, const void *v, const void *o, const void *dout,
                   const float *lse, void *dq, void *dk, void *dv, void *workspace,
                   size_t workspace_bytes, int B, int H, int H_kv, int N, int d, int dtype,
                   float scale, int causal, const uint8_t *block_mask, float p_drop,
                   unsigned long long seed, unsigned long long offset, void *stream);

/*
 * The three stages of fa_bwd, exposed so a caller (or a profiler) can order or time them.
 * fa_bwd_preprocess: delta[b,h,i] = sum_k dout[b,h,i,k] * o[b,h,i,k] in fp32 (FlashAttention-2
 *   reading notes, Algorithm 2, precomputation; FlashAttention paper detail, "Technique 2").
 * fa_bwd_dkdv: dK, dV for every key tile from q, k, v, dout, lse and delta.
 * fa_bwd_dq:   dQ for every query tile from q, k, v, dout, lse and delta.
 */
int fa_bwd_preprocess(const void *o, const void *dout, float *delta, int B, int H, int N, int d,
                      int dtype, void *stream);
int fa_bwd_dkdv(const void *q, const void *k, const void *v, const void *dout, const float *lse,
                const float *delta, void *dk, void *dv, int B, int H, int N, int d, int dtype,
                float scale, int causal, const uint8_t *block_mask, void *stream);
int fa_bwd_dq(const void *q, const void *k, const void *v, const void *dout, const float *lse,
              const float *delta, void *dq, int B, int H, int N, int d, int dtype, float scale,
              int causal, const uint8_t *block_mask, void *stream);

/*
 * Backward that allocates nothing: the same computation, arguments and results as fa_bwd,
 * without the workspace.  The pages have no counterpart; this entry point serves callers that
 * cannot allocate device memory themselves, such as a plug-in that a host application hands
 * only its input and output buffers while the application owns every device allocation, or
 * code on a latency-critical path where cudaMalloc's implicit device-wide synchronisation is
 * not acceptable.
 *
 * The D scratch lives in a fixed array compiled into libfa.so: FA_NOALLOC_MAX_ROWS floats
 * (4 MiB) that every GPU which loads the library keeps until the process exits.
 *  - Returns FA_ERR_INVALID, launching nothing, when B * H * N > FA_NOALLOC_MAX_ROWS, or
 *    when the block mask is wider than fa_bwd allows.
 *  - The first call on a device looks up the array's device address with that device current;
 *    make that first call before any stream capture.
 *  - Every call on a device uses the same array, which keeps the last call's values.  Calls
 *    that overlap on the GPU (other streams, other host threads) race on it and corrupt each
 *    other's gradients: order them.  Nothing in it has to start at zero, since each call
 *    writes every value it later reads.
 *  - Neither the call nor its set-up calls cudaMalloc, cudaFree or any allocating routine.
 */
#define FA_NOALLOC_MAX_ROWS (1u << 20)
int fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o, const void *dout,
                   const float *lse, void *dq, void *dk, void *dv, int B, int H, int N, int d,
                   int dtype, float scale, int causal, const uint8_t *block_mask, void *stream);

/*
 * Decode: a few new query rows per sequence against a KV cache.  FlashAttention-2 reading
 * notes, section on the KV cache (a 1 x d query per generated token against the N cached keys);
 * key ranges of the cache are processed by separate CTAs and merged with the statistic merge of
 * the FlashAttention paper detail, Technique 1.  The kernel is bound by reading K and V.
 *   q, o    : [B,H,Nq,d] (device), Nq >= 1 new rows per sequence;  lse : [B,H,Nq] fp32.
 *   k, v    : [B,H_kv,Nk,d] cache (device), Nk = its capacity; H_kv divides H and query head h
 *             reads K/V head h / (H / H_kv) (as fa_fwd_gqa).
 *   kv_len  : device int32 [B], the number of valid cached positions of each sequence (values
 *             are clamped to [0, Nk]), or NULL for Nk everywhere.
 *   causal  : 0: every new row sees all kv_len[b] keys.  != 0: the new rows are the last Nq
 *             positions of the sequence, row r is position kv_len[b] - Nq + r and sees keys
 *             j <= that position.  A row that sees no key gets O = 0 and LSE = -inf.
 *   workspace, workspace_bytes : device scratch of fa_decode_workspace_bytes() bytes,
 *             16-byte aligned (may be NULL when that is 0): the per-range partial results.
 * Errors as fa_fwd; B*H*Nq and B*H_kv*Nk must be below 2^31.
 */
size_t fa_decode_workspace_bytes(int B, int H, int H_kv, int Nq, int Nk, int d);
int fa_decode(const void *q, const void *k, const void *v, void *o, float *lse,
              const int *kv_len, int B, int H, int H_kv, int Nq, int Nk, int d, int dtype,
              float scale, int causal, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Synchronises `stream`, then returns and clears the current device's status word:
 * FA_OK, FA_ERR_TIMEOUT (a kernel gave up on a pipeline wait and returned early; its outputs
 * are undefined), FA_ERR_INTERNAL (a kernel refused to run on a misaligned shared-memory base;
 * its outputs are undefined) or FA_ERR_CUDA (the stream reported an error).
 */
int fa_sync_status(void *stream);

/* Static string naming a return code. */
const char *fa_status_string(int code);

/*
 * Test and diagnostics hooks (process-wide; they affect launches made after the call).
 * fa_debug_set_visit_log: when buf != NULL, every kernel ORs a bit into
 *   buf[((b*H + h) * T + i) * T + j] for each score tile (query tile i, key tile j) it
 *   computes: bit 0 forward, bit 1 dK/dV, bit 2 dQ.  bytes must cover B*H*T*T of the launches
 *   that follow, rounded up to a multiple of 4 (the bits are set by 32-bit atomic ORs); buf
 *   must be 4-byte aligned (otherwise FA_ERR_INVALID).  NULL (or bytes = 0) turns logging off.
 * fa_debug_set_wait_limit_ns: bound on every device pipeline wait (default 2 s; 0 restores it).
 * fa_debug_set_fault: 0 = none; 1 = the forward's load warp skips the first key tile of each
 *   CTA; 2 = the dK/dV pass's load warp skips its first Q tile; 3 = the dQ pass's load warp
 *   skips its first K tile.  The bounded waits then run out, the kernel returns early and
 *   fa_sync_status() reports FA_ERR_TIMEOUT; other values: FA_ERR_INVALID.
 * fa_debug_set_dkdv_splits: 0 = automatic; s > 0 splits every K/V head's query group of
 *   fa_bwd_gqa over min(s, H / H_kv) dK/dV CTAs per key tile (changes the workspace size).
 *   Negative: FA_ERR_INVALID.
 */
int fa_debug_set_visit_log(uint8_t *buf, size_t bytes);
int fa_debug_set_wait_limit_ns(unsigned long long ns);
int fa_debug_set_fault(int mode);
int fa_debug_set_dkdv_splits(int splits);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
