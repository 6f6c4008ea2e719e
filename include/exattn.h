/*
 * exattn.h -- C ABI of libexattn.so: exact fused scaled-dot-product
 * attention for NVIDIA GB300 (sm_103a).
 *
 * The operation ("Fused Kernel Compiler" page, subsection FlashAttention
 * Integration, equation Attention(Q,K,V) = softmax(QK^T / sqrt(d_k)) V):
 *
 *     s_ij  = scale * <q_i, k_j>, with s_ij = -inf where the causal mask
 *             hides key j;
 *     o_i   = sum_j softmax_j(s_i.) v_j;
 *     lse_i = log sum_j exp(s_ij)              (natural logarithm).
 *
 * It is computed in one pass with an online (running) softmax, so the score
 * and probability matrices never exist in device memory (same subsection,
 * items 1-4; "Kernel Fusion, Softmax, and Attention" page, attention
 * paragraph).  Results equal the definition up to floating-point rounding
 * order ("Optimizing LLM Inference ..." page, section The Shift Toward
 * Efficient Inference Architectures).
 *
 * Conventions shared by every entry point:
 *   - q, k, v, out, caches: bf16 (IEEE bfloat16), row-major, device memory,
 *     base addresses 16-byte aligned.  lse: fp32, device memory.
 *   - GQA: query head hq reads key/value head hq / (Hq / Hkv); Hq must be a
 *     multiple of Hkv.
 *   - Causal mask, aligned bottom-right: query row i sees key j iff
 *     j <= i + (Nk - Nq).  A row that sees no key gets o = 0, lse = -inf.
 *   - d (head dimension) is 64 or 128.  scale must be finite and > 0
 *     (callers usually pass 1/sqrt(d)).
 *   - stream is a cudaStream_t (NULL = legacy default stream).  Every call
 *     is asynchronous on that stream: validation happens on the host before
 *     anything is enqueued; nothing synchronises.
 *   - Ownership: the caller owns every buffer.  The library allocates no
 *     device memory per call; it keeps one 4-byte device status word per
 *     GPU (a static device variable) and a host-side cache of TMA tensor
 *     descriptors.
 *   - Errors: a non-zero return means nothing was launched (except
 *     EXATTN_ERR_CUDA, returned when a launch itself failed).  Faults found
 *     on the device (a bounded wait that ran out, a block-table entry out of
 *     range) never trap: the kernel records them in the status word and
 *     returns; read them with attn_get_device_status().
 */
#ifndef EXATTN_H_
#define EXATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  EXATTN_OK = 0,
  EXATTN_ERR_INVALID_ARG = 1, /* null pointer, negative size, Hq % Hkv != 0, bad scale */
  EXATTN_ERR_UNSUPPORTED = 2, /* d not in {64,128}, block_size != 16, size beyond limits */
  EXATTN_ERR_ALIGNMENT = 3,   /* a device pointer not 16-byte aligned */
  EXATTN_ERR_WORKSPACE = 4,   /* decode workspace missing or too small */
  EXATTN_ERR_CUDA = 5,        /* a CUDA runtime/driver call or launch failed */
  EXATTN_ERR_TIMEOUT = 6,     /* a bounded device wait ran out (reported as EXATTN_DEVICE_TIMEOUT_BIT) */
  EXATTN_ERR_DEVICE_BOUNDS = 7 /* table entry / ctx_len out of range (EXATTN_DEVICE_BOUNDS_BIT) */
} exattn_status;

/* Device status word bits (attn_get_device_status). */
#define EXATTN_DEVICE_TIMEOUT_BIT (1u << 0)
#define EXATTN_DEVICE_BOUNDS_BIT (1u << 1)

/*
 * Prefill attention (causal or not, with GQA).
 *   q    [B, Hq,  Nq, d] bf16      k, v [B, Hkv, Nk, d] bf16
 *   out  [B, Hq,  Nq, d] bf16      lse  [B, Hq, Nq] fp32, may be NULL
 * B, Hq, Hkv >= 1; Nq, Nk >= 0 (Nq == 0 or B == 0 is a no-op; Nk == 0
 * gives o = 0, lse = -inf).  Nq, Nk <= 2^30; B*Hq, B*Hkv <= 2^31 - 1.
 * Computes exactly one kernel launch.  Deterministic (no atomics on
 * outputs).
 */
int attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B, int Hq,
             int Hkv, int Nq, int Nk, int d, float scale, int causal, void* stream);

/*
 * Bytes of caller-provided device workspace attn_decode_paged needs: the
 * split-KV partial outputs (fp32 [num_seqs, Hq, max_splits, d]) and their
 * log-sum-exps (fp32 [num_seqs, Hq, max_splits]), where max_splits =
 * ceil(max_blocks_per_seq * block_size / split_tokens).  Returns 0 for
 * invalid arguments.
 */
size_t attn_decode_workspace_bytes(int num_seqs, int Hq, int d, int max_blocks_per_seq,
                                   int block_size);

/*
 * One-token decode over a block-paged KV cache ("Optimizing LLM Inference
 * ..." page, section Paged Attention and Dynamic KV Cache Management: the
 * cache is cut into fixed-size blocks and a block table maps each
 * sequence's logical token order to physical blocks).
 *   q        [num_seqs, Hq, d] bf16 (one query token per sequence)
 *   k_cache, v_cache [num_blocks, Hkv, block_size, d] bf16
 *   block_table int32 [num_seqs, max_blocks_per_seq]: physical block of
 *            logical block b of sequence s (entries past the last used
 *            block are not read)
 *   ctx_lens int32 [num_seqs]: cached tokens of sequence s, the current
 *            token included; all of them are visible (no mask)
 *   out      [num_seqs, Hq, d] bf16;  lse [num_seqs, Hq] fp32, may be NULL
 *   workspace/workspace_bytes: device scratch of at least
 *            attn_decode_workspace_bytes(...) bytes, 16-byte aligned;
 *            its contents need not be initialised and are clobbered.
 * block_size must be 16.  The key/value sweep of each sequence is cut into
 * splits of 512 tokens, or of 1024 when num_seqs * Hkv * ceil(Hq/Hkv/16) *
 * ceil(max_blocks_per_seq * 16 / 1024) is at least 8 * the SM count (the
 * longer split keeps every SM busy there and costs less fixed work per
 * byte); each split yields a partial output and log-sum-exp, and a second
 * kernel merges them (exact up to rounding).  The workspace is sized for
 * 512-token splits either way.
 * Two kernel launches; one when max_blocks_per_seq * block_size <= 512 (no
 * sequence can have a second split, so the split kernel writes the result
 * and no merge runs; same bits).  num_blocks >= 1.  A ctx_len of 0 gives o = 0, lse = -inf; a
 * ctx_len above max_blocks_per_seq * block_size or a table entry outside
 * [0, num_blocks) is clamped/skipped and flagged in the device status word.
 */
int attn_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_table, const int32_t* ctx_lens, void* out, float* lse,
                      int num_seqs, int Hq, int Hkv, int d, int block_size, int num_blocks,
                      int max_blocks_per_seq, float scale, void* workspace, size_t workspace_bytes,
                      void* stream);

/* Size of the static device scratch behind attn_decode_paged_static. */
#define EXATTN_STATIC_SCRATCH_BYTES (32u << 20)

/*
 * attn_decode_paged for callers that cannot allocate device memory.
 * (The pages have no counterpart: this is a deployment convenience.)
 *
 * Some callers may not call cudaMalloc at all: a plugin hosted inside an
 * inference server whose own pool owns every byte of device memory, or a
 * latency-critical decode loop where cudaMalloc's implicit device-wide
 * synchronisation is not allowed.  This entry point takes the same
 * arguments as attn_decode_paged minus the workspace; its split-KV scratch
 * is a file-scope static device array of EXATTN_STATIC_SCRATCH_BYTES (32 MiB)
 * that every GPU which loads the library holds until the process exits.
 * The caller still passes every input and output buffer.
 *
 * - Limit: when attn_decode_workspace_bytes(num_seqs, Hq, d,
 *   max_blocks_per_seq, block_size) exceeds EXATTN_STATIC_SCRATCH_BYTES the
 *   call returns EXATTN_ERR_WORKSPACE and launches nothing.  For example
 *   64 sequences x 32 query heads at d = 128 with block tables of up to
 *   8192 tokens need about 16 MiB and fit; use attn_decode_paged beyond
 *   the limit.
 * - No allocation: it calls no cudaMalloc/cudaFree or allocating library.
 * - Set-up: the first call on a device, with that device current, looks up
 *   the array's device address once (cudaGetSymbolAddress); make that first
 *   call before any stream capture.
 * - Sharing: every call on a device uses the same array, and the array
 *   keeps the last call's contents.  Nothing in it needs to start at zero
 *   (each split's partial result is written before it is read), but calls
 *   whose executions overlap on the GPU (different streams, or several host
 *   threads) race on it; serialise them on one stream.
 */
int attn_decode_paged_static(const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_table, const int32_t* ctx_lens, void* out,
                             float* lse, int num_seqs, int Hq, int Hkv, int d, int block_size,
                             int num_blocks, int max_blocks_per_seq, float scale, void* stream);

/*
 * Residual add + RMS normalisation, the fusion that sits next to attention
 * in every layer ("Inference Engineering VII.07: Kernel and Operator
 * Fusion" page, section 4: the fused kernel loads x and the residual once,
 * adds, reduces the sum of squares, scales, and stores both results;
 * section 5: the sum is returned because the next layer's residual add
 * needs it).  For each of n_rows rows of `hidden` values:
 *   residual_out = x + residual
 *   out          = residual_out * rsqrt(mean(residual_out^2) + eps) * weight
 * with the sum, the mean of squares and the products in fp32 and each
 * output rounded once to bf16 (nearest even).
 *   x, residual, out, residual_out  [n_rows, hidden] bf16, row-major
 *   weight                          [hidden] bf16
 * hidden must be a multiple of 8 in [8, 16384]; eps finite and >= 0;
 * n_rows >= 0 (0 launches nothing; pointers may then be NULL).  Every
 * pointer 16-byte aligned.  out and residual_out may each be the same
 * pointer as x or residual (in place), but not each other and not weight;
 * no other overlap is allowed.  The caller owns every buffer.  One kernel
 * launch on `stream`, asynchronous; deterministic.
 */
int attn_add_rms_norm(const void* x, const void* residual, const void* weight, void* out,
                      void* residual_out, int n_rows, int hidden, float eps, void* stream);

/*
 * Bytes of caller-provided device workspace attn_bwd needs: fp32
 * (lse * log2 e, D) pairs per query row ([B*Hq][Nq rounded up to even][2])
 * and, when query heads share a KV head (Hq > Hkv), room for fp32 dK and dV
 * partials per query head ([2][B*Hq][Nk][d], placed on the next 32-byte
 * boundary: 16 bytes of slack).
 * Returns 0 for invalid arguments (or nothing to store).
 */
size_t attn_bwd_workspace_bytes(int B, int Hq, int Hkv, int Nq, int Nk, int d);

/*
 * Attention backward: the gradients of attn_fwd's output with respect to
 * q, k and v, given dout ("Kernel Fusion, Softmax, and Attention" page:
 * training runs a different schedule of the same attention equation).  With
 * P = softmax(scale * q k^T + mask) rebuilt from the forward's lse:
 *   D_i  = <dout_i, out_i>,  dS = P * (dout v^T - D),
 *   dv = P^T dout,  dk = scale dS^T q,  dq = scale dS k,
 * dk, dv summed over the query heads of each KV head.
 *   q, out, dout, dq [B, Hq, Nq, d] bf16;  k, v, dk, dv [B, Hkv, Nk, d] bf16
 *   lse [B, Hq, Nq] fp32: attn_fwd's log-sum-exp for the same inputs
 *   workspace: attn_bwd_workspace_bytes(...) bytes, 16-byte aligned (its
 *   contents need not be initialised and are clobbered)
 * scale, causal (same bottom-right mask), d and the head counts as attn_fwd;
 * B*Hq, B*Hkv <= 65535 and Nq, Nk <= 65535 * 64 (EXATTN_ERR_UNSUPPORTED
 * beyond).  All tensor pointers 16-byte aligned (lse 4); the tensors of an
 * empty side may be NULL (q, out, dout, lse, dq when Nq == 0; k, v, dk, dv
 * when Nk == 0: the other side's gradients are then zero); no output may
 * overlap an input.  B == 0 or Nq == Nk == 0 launches nothing.
 * Two or three kernel launches on `stream`: dq (which also forms D) and
 * dk/dv on the tensor cores, each a persistent grid of at most one CTA per
 * SM; when query heads share a KV head, each writes fp32 partials to the
 * workspace and a third kernel sums them.  The second and third are
 * programmatic dependent launches (they may start as the previous launch
 * drains).  Asynchronous,
 * deterministic (no atomics; sums in head order).  A bounded wait inside the
 * kernels that runs out sets EXATTN_DEVICE_TIMEOUT_BIT.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
             const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk,
             int d, float scale, int causal, void* workspace, size_t workspace_bytes, void* stream);

/*
 * CUDA-graph capture of one decode step ("Optimizing LLM Inference ..."
 * page, section Compilation and CUDA Graphs: a captured sequence of
 * launches is replayed with one call, removing per-launch overhead).
 * attn_decode_graph_capture records exactly the work attn_decode_paged
 * would enqueue for these arguments (split kernel + merge) on a private
 * stream and instantiates it; nothing runs.  The graph keeps every pointer
 * and size it was captured with: the caller keeps those buffers alive and
 * may change their contents (q, ctx_lens, block_table, the caches) between
 * launches; ctx_lens entries must stay <= max_blocks_per_seq * 16.  Same
 * argument rules and errors as attn_decode_paged, plus num_seqs >= 1 and a
 * non-NULL graph_out (set to NULL on failure).  The graph belongs to the
 * device current at capture.
 * attn_graph_launch enqueues one replay on `stream` (asynchronous).
 * attn_graph_destroy frees the graph (NULL is a no-op); no replay may still
 * be pending.
 */
typedef struct exattn_graph exattn_graph;

int attn_decode_graph_capture(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_table, const int32_t* ctx_lens, void* out,
                              float* lse, int num_seqs, int Hq, int Hkv, int d, int block_size,
                              int num_blocks, int max_blocks_per_seq, float scale, void* workspace,
                              size_t workspace_bytes, exattn_graph** graph_out);
int attn_graph_launch(exattn_graph* graph, void* stream);
int attn_graph_destroy(exattn_graph* graph);

/*
 * Rotary position embedding of the new tokens' queries and keys, then the
 * store of each token's rotated key and its value into the block-paged
 * cache, in one kernel ("Inference Engineering VII.07: Kernel and Operator
 * Fusion" page, section 2, "rope + cache write: RoPE then KV store";
 * "Fused Kernel Compiler" page, table of fusion patterns, "RoPE
 * embedding: sin, cos, rotate").  Pairs (i, i + d/2) of every head vector
 * of token t turn by theta_i = positions[t] * base^(-2i/d):
 *   y_i = x_i cos theta_i - x_(i+d/2) sin theta_i
 *   y_(i+d/2) = x_(i+d/2) cos theta_i + x_i sin theta_i
 * (angles reduced modulo 2 pi exactly in 64-bit fixed point from
 * frequencies formed in fp64, rotation in fp32, one bf16 rounding).
 *   q        [num_tokens, Hq, d] bf16: rotated in place
 *   k, v     [num_tokens, Hkv, d] bf16: read only
 *   seq_ids, positions int32 [num_tokens]: sequence and 0-based position of
 *            each token
 *   block_table int32 [num_seqs, max_blocks_per_seq] (as attn_decode_paged)
 *   k_cache, v_cache [num_blocks, Hkv, 16, d] bf16: token t's rotated key
 *            and its value go to slot positions[t] % 16 of physical block
 *            block_table[seq][positions[t] / 16]; nothing else is written.
 * d a multiple of 16 in [16, 256], (Hq + 3 Hkv) * d / 16 <= 2048 (e.g. up to
 * 128 query and 32 key/value heads at d = 128); base finite and > 1; num_seqs,
 * num_blocks, max_blocks_per_seq >= 1; num_tokens >= 0 (0 launches
 * nothing).  q, k, v and the caches 16-byte aligned, the int32 arrays
 * 4-byte aligned; k_cache != v_cache; no other overlap.  Two tokens that
 * map to the same slot race.  A token whose sequence, position or table
 * entry lies outside the table or the cache is rotated in q but stores
 * nothing, and sets EXATTN_DEVICE_BOUNDS_BIT.  One kernel launch on
 * `stream`, asynchronous.
 */
int attn_rope_cache_write(void* q, const void* k, const void* v, const int32_t* seq_ids,
                          const int32_t* positions, const int32_t* block_table, void* k_cache,
                          void* v_cache, int num_tokens, int Hq, int Hkv, int d, int num_seqs,
                          int num_blocks, int max_blocks_per_seq, float base, void* stream);

/*
 * Synchronises `stream`, then reads and clears the status word of the
 * current device and stores it in *status_out: 0, or an OR of
 * EXATTN_DEVICE_*_BIT (the bits are small, so the value is never negative).
 * status_out must not be NULL (EXATTN_ERR_INVALID_ARG).  Returns EXATTN_OK
 * or EXATTN_ERR_CUDA.
 */
int attn_get_device_status(void* stream, int* status_out);

/* Human-readable name of an exattn_status value (static string). */
const char* attn_status_string(int status);

/* Split granularity, in tokens, that attn_decode_workspace_bytes sizes the
 * workspace for (512; attn_decode_paged may use splits of twice that). */
int attn_decode_split_tokens(void);

/*
 * Diagnostic for the failure path.  Launches one CTA that waits, through the
 * same bounded mbarrier wait the attention kernels use, on a barrier that
 * nothing ever completes.  After budget_ns nanoseconds (1 .. 10^10) the wait
 * gives up, the kernel sets EXATTN_DEVICE_TIMEOUT_BIT in the status word and
 * returns; the GPU context stays usable.  Returns EXATTN_OK once launched.
 */
int attn_debug_expire_wait(unsigned long long budget_ns, void* stream);

/* Drops the host-side descriptor cache.  Safe to call at any time when no
 * other thread is inside the library. */
void attn_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* EXATTN_H_ */
