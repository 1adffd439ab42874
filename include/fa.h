/*
 * fa.h - exact scaled-dot-product attention for one NVIDIA GB300 (sm_103a).
 *
 * O = softmax(scale * Q K^T [+ mask]) V, computed FlashAttention-style: the
 * N x N score matrix S and probability matrix P never reach device memory.
 * The forward keeps a running row maximum m, row sum l and unnormalised
 * output O~ per query row and updates them block by block with the online
 * softmax recurrence ("注意力为什么受限于显存带宽：用算术强度与分块把
 * FlashAttention 推导清楚", section 六; "4. FlashAttention 深度剖析",
 * sections 4.2.2-4.2.4 and 4.3.2); it saves the per-row log-sum-exp
 * L = m + log l, from which the backward recomputes P (same pages, section
 * 八 and section 4.3.4).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Tensors are caller-owned DEVICE memory.  Q, K, V, O, dO, dQ, dK, dV are
 *   bf16 (__nv_bfloat16 bit patterns), contiguous [B, H, N, d] (d fastest),
 *   each base address 16-byte aligned.  LSE is fp32 [B, H, N].
 * - Supported head dimensions: d = 64, 128, 256.  B, H, N >= 1 and
 *   B*H*N*d < 2^31 elements per tensor.
 * - scale multiplies Q K^T; it must be finite and > 0 (1/sqrt(d) is usual).
 * - causal != 0 masks key j for query i when j > i (0-based; N queries and
 *   N keys).
 * - kv_len is NULL (no padding) or a DEVICE pointer to int32[B]: keys
 *   j >= kv_len[b] are masked for every query of batch b.  Values are
 *   clamped to [0, N]; a query row that sees no key at all gets O = 0 and
 *   LSE = -inf (its gradients are 0).
 * - stream is a cudaStream_t passed as void* (NULL = legacy default
 *   stream).  Every call only enqueues work and returns; nothing here
 *   synchronises except fa_check().  The library never allocates memory.
 * - Outputs are fully overwritten.
 * - Errors: FA_ERR_INVALID_ARG (null or misaligned pointer, bad size,
 *   scale not finite or <= 0, workspace too small), FA_ERR_UNSUPPORTED (head
 *   dimension, or a GPU that is not sm_103), FA_ERR_CUDA (a CUDA call or
 *   kernel launch failed; cudaGetLastError() holds the detail).  Argument
 *   errors are reported before anything is enqueued.
 * - Kernels never spin forever: every wait inside them gives up after about
 *   two seconds, records FA_ERR_TIMEOUT in a per-device status word and
 *   returns; fa_check() reports and clears it.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,
  FA_ERR_UNSUPPORTED = 2,
  FA_ERR_CUDA = 3,
  FA_ERR_TIMEOUT = 4
} fa_status_t;

/*
 * Forward.  Writes O = softmax(scale*QK^T + mask) V (bf16 [B,H,N,d]) and
 * LSE_i = ln sum_j exp(scale*q_i.k_j) over the visible keys (fp32 [B,H,N],
 * natural log, the statistic L = m + log l of "4. FlashAttention 深度剖析"
 * section 4.3.2).  Tiling and the online update follow section 4.3.2 of
 * that page with the loop order "outer over Q tiles" of its section 4.4.3;
 * key blocks entirely above the causal diagonal are skipped (section 4.3.2,
 * last note).
 */
fa_status_t fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                   int B, int H, int N, int d, float scale, int causal,
                   const int* kv_len, void* stream);

/*
 * Bytes of device workspace fa_bwd needs for these sizes: the fp32 row
 * statistics D = rowsum(dO o O) and LSE*log2(e), each [B*H, Npad] with Npad =
 * N rounded up to 128, and the fp32 dQ accumulator of B*H*Npad*d elements
 * ([B*H, Npad, d] for d = 64, [B*H, d, Npad] for d = 128 and 256), and
 * Npad/128 uint32 for the key blocks' schedule order (written when a block
 * mask comes without its host copy); each region starts on a 256-byte
 * boundary.  Returns 0 for invalid sizes.
 */
size_t fa_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * Backward by recomputation ("注意力为什么受限于显存带宽…" section 八;
 * "4. FlashAttention 深度剖析" section 4.3.4): P is rebuilt on chip from
 * Q, K and the saved LSE (P_ij = exp(scale*q_i.k_j - LSE_i)); then
 *   D = rowsum(dO o O),  dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),
 *   dQ = scale * dS K,   dK = scale * dS^T Q.
 * Inputs q, k, v, o, dO (bf16 [B,H,N,d]) and lse (fp32 [B,H,N], as written
 * by fa_fwd with the same scale, causal and kv_len).  Outputs dq, dk, dv
 * (bf16 [B,H,N,d]).  workspace: caller-owned device memory of at least
 * fa_bwd_workspace_bytes(B,H,N,d) bytes, 256-byte aligned; its contents on
 * entry do not matter and on return are unspecified.  dQ is summed over the
 * key blocks in fp32 by bulk reduce-adds that the L2 performs in an order
 * that varies, so its last bits can differ from run to run; dK and dV are
 * each accumulated by one SM and repeat bit for bit.
 */
fa_status_t fa_bwd(const void* q, const void* k, const void* v, const void* o,
                   const void* dO, const float* lse, void* dq, void* dk, void* dv,
                   int B, int H, int N, int d, float scale, int causal, const int* kv_len,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * The three launches fa_bwd makes, callable one by one (same workspace, same
 * stream order); fa_bwd is exactly fa_bwd_prep, fa_bwd_dkdv, fa_bwd_dq.
 *
 * fa_bwd_prep: D_i = rowsum(dO o O)_i and LSE_i * log2(e) into the workspace
 *   (padded to a multiple of 128 rows), and zeroes the fp32 dQ accumulator.
 * fa_bwd_dkdv: recomputes P per 128x128 tile from Q, K and the saved LSE,
 *   writes dK and dV (bf16) and adds dS K into the fp32 dQ accumulator;
 *   needs fa_bwd_prep to have run on this workspace.
 * fa_bwd_dq:   dQ = bf16(scale * accumulator); needs fa_bwd_dkdv.
 * Argument rules and errors are those of fa_bwd for the arguments each takes.
 */
fa_status_t fa_bwd_prep(const void* o, const void* dO, const float* lse, int B, int H, int N,
                        int d, void* workspace, size_t workspace_bytes, void* stream);
fa_status_t fa_bwd_dkdv(const void* q, const void* k, const void* v, const void* dO, void* dk,
                        void* dv, int B, int H, int N, int d, float scale, int causal,
                        const int* kv_len, void* workspace, size_t workspace_bytes,
                        void* stream);
fa_status_t fa_bwd_dq(void* dq, int B, int H, int N, int d, float scale, void* workspace,
                      size_t workspace_bytes, void* stream);

/*
 * Attention variants: grouped K/V heads and a sliding window.
 *
 * h_kv: K/V heads.  K, V, dK, dV are bf16 [B, h_kv, N, d] and query head h
 *   reads K/V head h / (H / h_kv); 1 <= h_kv <= H and H % h_kv == 0.
 *   h_kv = H is multi-head attention, h_kv = 1 multi-query attention, values
 *   in between grouped-query attention, as FlashAttention-2 supports them
 *   ("注意力为什么受限于显存带宽…" section 九; "炉案与百步之外的仓库：Flash
 *   Attention 与注意力计算的工艺极限" section 六).
 * window_left, window_right: flash-attn's window_size=(left, right) (same
 *   section 六; "4. FlashAttention 深度剖析" 4.8.1).  -1 leaves that side
 *   unbounded; otherwise query i sees key j only when
 *   i - window_left <= j <= i + window_right.  The window combines with
 *   causal and kv_len; a row may then see no key at all (O = 0, LSE = -inf).
 *   Key blocks outside every row's window are skipped, not masked
 *   ("深入浅出 FlashAttention：快如闪电的精确注意力机制与 IO 感知计算"
 *   第八部分).
 * block_mask: NULL, or device memory holding a row-major [T, T] byte matrix
 *   with T = ceil(N / 128), shared by every batch entry and head.  Entry
 *   (a, b) zero hides keys 128b .. 128b+127 from queries 128a .. 128a+127:
 *   the coarse block-level mask of Block-Sparse FlashAttention
 *   ("深入浅出 FlashAttention…" 第八部分).  The kernels skip such blocks
 *   (neither load nor compute them).  It combines with causal, the window
 *   and kv_len; a row may then see no key (O = 0, LSE = -inf).  With a block
 *   mask, tiles are scheduled one per unit instead of in causal pairs.  The
 *   caller keeps the mask unchanged until the call's work has run.  fa_decode
 *   rejects a block mask (FA_ERR_UNSUPPORTED).
 * block_mask_host: NULL, or host memory holding the same T * T bytes as
 *   block_mask (ignored when block_mask is NULL).  The call reads it before
 *   it returns, on the calling thread, to balance its persistent schedule:
 *   a tile's work is its count of computed blocks, and the last heads' tiles
 *   go, most work first, to the least-loaded SMs.  The results do not depend
 *   on it; a copy that differs from block_mask only unbalances the schedule.
 *   NULL (and no causal flag): the kernels plan the schedule on the device
 *   from block_mask: the tiles (the backward's key blocks) are sorted by
 *   their computed blocks, most first, and dealt over the SMs in rounds that
 *   turn direction, which leaves the busiest SM some 8 % above the mean on
 *   an uneven mask (about 2 % with the host copy).  Past 256 tiles
 *   (forward) or 1024 key blocks (backward) they go round-robin instead,
 *   which with an uneven mask can leave some SMs with a third more work
 *   than the mean.
 * A NULL variant pointer means {H, -1, -1, NULL, NULL}; an aggregate
 * initialiser that stops after window_right (or block_mask) leaves the later
 * members NULL.
 */
typedef struct fa_variant {
  int h_kv;
  int window_left;
  int window_right;
  const unsigned char* block_mask;
  const unsigned char* block_mask_host;
} fa_variant_t;

/*
 * fa_fwd and fa_bwd for a variant; every other argument is as in fa_fwd and
 * fa_bwd, with K, V, dK, dV shaped [B, h_kv, N, d] and the workspace of
 * fa_bwd_workspace_bytes(B, H, N, d).  dK and dV are the sums over each
 * group's query heads.  FA_ERR_INVALID_ARG also for h_kv not dividing H or a
 * window side below -1.  lse must come from fa_fwd_v with the same variant.
 */
fa_status_t fa_fwd_v(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int H, int N, int d, float scale, int causal,
                     const int* kv_len, const fa_variant_t* variant, void* stream);
fa_status_t fa_bwd_v(const void* q, const void* k, const void* v, const void* o,
                     const void* dO, const float* lse, void* dq, void* dk, void* dv,
                     int B, int H, int N, int d, float scale, int causal, const int* kv_len,
                     const fa_variant_t* variant, void* workspace, size_t workspace_bytes,
                     void* stream);

/* fa_bwd_dkdv for a variant (fa_bwd_v is fa_bwd_prep, fa_bwd_dkdv_v, fa_bwd_dq). */
fa_status_t fa_bwd_dkdv_v(const void* q, const void* k, const void* v, const void* dO, void* dk,
                          void* dv, int B, int H, int N, int d, float scale, int causal,
                          const int* kv_len, const fa_variant_t* variant, void* workspace,
                          size_t workspace_bytes, void* stream);

/*
 * Split-KV decoding: Nq new queries per head against a long key/value cache
 * (FlashDecoding, "4. FlashAttention 深度剖析" 4.8.3).  The keys of every K/V
 * head are cut into `splits` chunks that different SMs process at once; each
 * chunk yields a partial (O_s normalised by its own row sum, LSE_s), and a
 * second kernel merges the chunks with the associative rule of 4.2.4:
 *   LSE = log sum_s exp(LSE_s),   O = sum_s exp(LSE_s - LSE) O_s.
 *
 * q, o: bf16 [B, H, Nq, d]; k, v: bf16 [B, h_kv, Nk, d] (h_kv from the
 * variant, H when NULL); lse: fp32 [B, H, Nq].  kv_len: NULL (every entry has
 * Nk valid keys) or a device int32[B] of cache lengths, clamped to [0, Nk].
 * Query t of batch entry b is the token at position kv_len[b] - Nq + t:
 * with causal it sees keys j <= that position, the variant's window is taken
 * around it, and keys j >= kv_len[b] are never seen.  A query that sees no
 * key gets O = 0, LSE = -inf.  The query heads of one K/V head are processed
 * together: (H / h_kv) * Nq must be at most 128 (else FA_ERR_UNSUPPORTED).
 * workspace: device memory of fa_decode_workspace_bytes(B, H, Nq, d, splits)
 * bytes, 256-byte aligned, for the fp32 partials.  splits >= 1; chunks are
 * whole 128-key blocks, so at most ceil(Nk / 128) chunks are used.
 * fa_decode_splits returns the library's choice for this GPU (0 for invalid
 * sizes): with fewer K/V heads (B * h_kv) than SMs, the most chunks of at
 * least 8 key blocks that run as one wave; otherwise the count whose units
 * fill the SMs' waves best.  Other arguments and errors as for fa_fwd_v.
 */
int fa_decode_splits(int B, int h_kv, int Nk);
size_t fa_decode_workspace_bytes(int B, int H, int Nq, int d, int splits);
fa_status_t fa_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                      int B, int H, int Nq, int Nk, int d, float scale, int causal,
                      const int* kv_len, const fa_variant_t* variant, int splits,
                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * FP8 (E4M3) forward ("4. FlashAttention 深度剖析" 4.5.4: E4M3 operands for
 * the forward, a scale per block applied at load, FP32 accumulation).
 *
 * Layouts, with nb = ceil(N / 128) and h_kv from the variant:
 *   q8  E4M3 [B, H, N, d]        q_scale fp32 [B, H, nb]     (per 128-row tile)
 *   k8  E4M3 [B, h_kv, N, d]     k_scale fp32 [B, h_kv, nb]  (per 128-key block)
 *   v8t E4M3 [B, h_kv, d, nb*128] (V transposed, keys padded with zeros)
 *                                v_scale fp32 [B, h_kv]      (per head)
 * A stored value x8 stands for x8 * scale.  d = 128 or 256 (64:
 * FA_ERR_UNSUPPORTED); E4M3 buffers 16-byte aligned.
 *
 * fa_fp8_quantize writes these from bf16 Q, K, V ([B,H,N,d], [B,h_kv,N,d]):
 * scale = amax / 448 of the block (1 for an all-zero block) and
 * x8 = E4M3(x * (448 / amax)), rounded to nearest even and saturated.
 *
 * fa_fwd_fp8 computes O (bf16 [B,H,N,d]) and LSE (fp32 [B,H,N]) from them:
 * S = (q8 k8^T) * q_scale * k_scale * scale on the tensor core in FP32; the
 * online softmax of fa_fwd over 128-key blocks.  A row's reference maximum m
 * starts at its first block's maximum and is raised to a block's maximum
 * only when that exceeds m by more than a factor 2^4, so P = exp(S - m) <=
 * 16; P enters the P V product as E4M3(16 P) <= 256 against v8t (FP32
 * accumulation), the row sum l adds the unrounded P, and O = v_scale *
 * (sum of E4M3(16 P) v8) / (16 l), LSE = m + ln l.  The result differs from
 * exact attention of the dequantised inputs (x8 * scale) only by E4M3's
 * rounding of P (2^-4 of a weight in E4M3's normal range, 2^-10 of the row's
 * largest weight below it) and FP32 rounding.  causal, kv_len and the
 * variant as for fa_fwd_v.
 */
fa_status_t fa_fp8_quantize(const void* q, const void* k, const void* v, int B, int H, int N,
                            int d, const fa_variant_t* variant, void* q8, float* q_scale,
                            void* k8, float* k_scale, void* v8t, float* v_scale, void* stream);
fa_status_t fa_fwd_fp8(const void* q8, const float* q_scale, const void* k8,
                       const float* k_scale, const void* v8t, const float* v_scale, void* o,
                       float* lse, int B, int H, int N, int d, float scale, int causal,
                       const int* kv_len, const fa_variant_t* variant, void* stream);

/*
 * Self-test of the bounded waits: enqueues one tiny kernel that waits on a
 * barrier nothing ever completes, with a limit of timeout_us microseconds
 * (1 .. 1000000) instead of the kernels' two seconds.  The wait gives up,
 * the kernel records FA_ERR_TIMEOUT in the status word and returns, so the
 * following fa_check() returns FA_ERR_TIMEOUT (and clears it) and the
 * device stays usable.  Returns FA_ERR_INVALID_ARG for a limit out of range.
 */
fa_status_t fa_selftest_wait_timeout(unsigned int timeout_us, void* stream);

/*
 * fa_bwd_noalloc: the backward pass for callers that cannot allocate device
 * memory.  Same arguments, results and errors as fa_bwd (checked in the same
 * order), minus the workspace:
 * the scratch fa_bwd needs (fa_bwd_workspace_bytes(B,H,N,d) bytes) comes from
 * a fixed array of FA_BWD_NOALLOC_MAX_SCRATCH_BYTES that the library keeps in
 * device memory, so this call allocates nothing.  It is meant for code that is
 * not allowed to allocate: an allocator or memory-pool hook that must not
 * re-enter itself, a plugin that is handed only its tensors, or a loop that
 * cannot take cudaMalloc's implicit synchronisation.
 *
 * - Sizes whose scratch exceeds the maximum return FA_ERR_INVALID_ARG before
 *   anything is enqueued (64 MiB covers, e.g., B*H*N*d up to about 16M
 *   elements).
 * - Every GPU that loads this part of the library holds the array until the
 *   process exits.  Its device address is looked up on the first call on each
 *   device that passes the argument checks (with that device current); make
 *   that first call before any stream capture.  A lookup that fails returns
 *   FA_ERR_CUDA, leaves no error pending in cudaGetLastError(), and is tried
 *   again by the next call.
 * - All calls share the array: calls whose kernels overlap on the GPU race
 *   and give wrong gradients.  Calls ordered on one stream are fine; each call
 *   re-initialises the scratch it reads, so no state carries over.
 * The pages describe no such variant; it exists only for such callers.
 */
#define FA_BWD_NOALLOC_MAX_SCRATCH_BYTES (64u * 1024u * 1024u)
fa_status_t fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                           const void* dO, const float* lse, void* dq, void* dk, void* dv,
                           int B, int H, int N, int d, float scale, int causal,
                           const int* kv_len, void* stream);

/*
 * Waits for `stream`, then reads and clears the current device's status
 * word.  FA_ERR_TIMEOUT if a kernel gave up waiting since the last check,
 * FA_ERR_CUDA if the stream reports an error, FA_OK otherwise.
 */
fa_status_t fa_check(void* stream);

/* Static, human-readable name of a status code. */
const char* fa_status_string(fa_status_t status);

/* Library version as major*10000 + minor*100 + patch.  1.1: fa_variant_t
 * gained block_mask (a trailing member, NULL in aggregate initialisers that
 * stop before it).  1.2: fa_variant_t gained block_mask_host (the same). */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
