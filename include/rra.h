/*
 * rra.h -- ragged (token-pruned) bidirectional attention for ViTs, C ABI.
 *
 * The operation is the pack -> attend -> unpack pipeline of "Dispatch-Aware
 * Ragged Attention for Pruned Vision Transformers" (arXiv 2604.15408):
 *   - abstract: a bidirectional (non-causal) attention kernel run on
 *     token-pruned ViT sequences (at most 197 tokens at 224 px, 577 at
 *     384 px) inside a complete pack-attend-unpack pipeline whose outputs
 *     match padded SDPA;
 *   - agents-report.net article on the paper, section "方法概覽：
 *     pack-attend-unpack 流程" (method overview): (1) fused token packing --
 *     GPU index work yields per-image offsets (cu_seqlens) and destination
 *     indices, and a vectorised copy gathers surviving tokens into one flat
 *     buffer; (2) the ragged attention kernel runs directly on that compact
 *     buffer; (3) unpack writes results back to the original batch positions
 *     using cu_seqlens.  Section "問題：填充與派遣的瓶頸" (problem) names host
 *     dispatch as the bottleneck, which the graph plan below addresses.
 *
 * Conventions for every entry point:
 *   - Tensors are device pointers (host pointers where an entry point says
 *     so: rra_pipeline_host, rra_pipeline_mapped), contiguous, 16-byte
 *     aligned (else RRA_ERR_MISALIGNED).  Padded tensors are [B, N, H, d] row-major; packed
 *     tensors are [cap, H, d] with cap = B*N rows, of which the first T (the
 *     number of kept tokens, known only on the device) are written.
 *   - d must be 64 (else RRA_ERR_UNSUPPORTED); 1 <= N <= 1024; H >= 1;
 *     1 <= B <= 65535; B*N*H*d < 2^31.
 *   - The keep mask is uint8 [B, N]; any nonzero byte keeps the token.
 *   - Input dtype is RRA_F16 or RRA_BF16; attention outputs may also be
 *     RRA_F32.  Softmax and both products accumulate in fp32.
 *   - Ownership: the caller allocates and frees every buffer.  The library
 *     allocates no device memory, except the CUDA graph owned by an rra_plan
 *     (and the fixed scratch array of rra_pipeline_static, which is part of
 *     the loaded module); rra_attend_wait keeps one 64-byte page-locked host
 *     word per device.
 *   - Asynchrony: every call only enqueues work on `stream` (a cudaStream_t;
 *     NULL is the legacy default stream).  Nothing synchronises and nothing
 *     is copied device->host, so the pack / attend / unpack / pipeline calls
 *     can be captured in a CUDA graph.  The exceptions block on purpose:
 *     rra_attend_wait, rra_get_device_error and the rra_time_* helpers.
 *   - Errors: argument checks run on the host before anything is launched
 *     and return a status with nothing enqueued.  A failed launch returns
 *     RRA_ERR_CUDA.  Inconsistent device-side data (e.g. a cu_seqlens entry
 *     longer than max_seqlen) never traps: the kernel skips the bad work and
 *     records a code that rra_get_device_error() reads after the caller syncs.
 *   - rra_last_error_message() gives a one-line description of the last
 *     non-OK status returned on the calling thread.
 */
#ifndef RRA_H
#define RRA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define RRA_API __attribute__((visibility("default")))
#else
#define RRA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RRA_OK = 0,
  RRA_ERR_INVALID_ARG = 1, /* null pointer, bad size, bad enum          */
  RRA_ERR_UNSUPPORTED = 2, /* valid but unsupported (d != 64, N > 1024)  */
  RRA_ERR_MISALIGNED = 3,  /* a tensor pointer not 16-byte aligned       */
  RRA_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed       */
  RRA_ERR_DEVICE = 5       /* a kernel recorded a device-side error code */
} rra_status;

typedef enum { RRA_F16 = 0, RRA_BF16 = 1, RRA_F32 = 2 } rra_dtype;

/* Device-side error codes reported by rra_get_device_error(). */
enum {
  RRA_DEVERR_NONE = 0,
  RRA_DEVERR_SEQ_TOO_LONG = 1,  /* attend: cu_seqlens[b+1]-cu_seqlens[b] > max_seqlen */
  RRA_DEVERR_SEQ_NEGATIVE = 2,  /* attend: cu_seqlens decreasing                      */
  RRA_DEVERR_INDEX_RANGE = 3,   /* attend/unpack: src_idx or dst_idx out of range     */
  RRA_DEVERR_WAIT_TIMEOUT = 4   /* a bounded on-chip wait gave up                     */
};

/* Bytes of workspace rra_pipeline needs for these sizes (0 on bad args):
 * cu_seqlens [B+1], dst_idx [B*N], src_idx [B*N] (int32), then packed Q, K, V
 * [B*N, H, d] in the input dtype, each section 256-byte aligned. */
RRA_API size_t rra_workspace_bytes(int B, int N, int H, int d, rra_dtype in_dtype);

/* Byte offsets of the sections of that workspace, in the order
 * cu_seqlens, dst_idx, src_idx, qp, kp, vp (6 entries). */
RRA_API rra_status rra_workspace_offsets(int B, int N, int H, int d, rra_dtype in_dtype,
                                         size_t offsets[6]);

/* Fused token packing (method overview, bullet 1), one kernel launch:
 *   cu_seqlens[b]   = number of kept tokens in images 0..b-1 (cu[B] = T);
 *   dst_idx[b*N+j]  = packed row of token (b, j), or -1 if it is pruned;
 *   src_idx[t]      = b*N+j for packed row t (t < T; rows >= T untouched);
 *   qp/kp/vp[t]     = bit copies of q/k/v[b, j] (all H heads of the token);
 *   out_zero_fill   = optional [B, N, H, d] tensor of `out_dtype`: its rows at
 *                     pruned positions are set to +0 (the unpack's fill, done
 *                     here so a scattering rra_attend completes the output).
 * Packed order is images in batch order, tokens in original order.  With
 * qp, kp and vp all NULL only the indices and the zero fill are produced
 * (q, k and v are then not read) -- the index pass of rra_pipeline. */
RRA_API rra_status rra_pack(const uint8_t* keep, int B, int N, int H, int d, rra_dtype in_dtype,
                            const void* q, const void* k, const void* v,
                            int32_t* cu_seqlens, int32_t* dst_idx, int32_t* src_idx,
                            void* qp, void* kp, void* vp,
                            void* out_zero_fill, rra_dtype out_dtype, void* stream);

/* Re-pack between the layers of progressive token pruning (EViT-like pruners
 * drop tokens at a few layers; abstract, both revisions): the next layer's
 * packed buffers are built from the previous layer's packed buffers instead
 * of padded tensors, so no padded tensor exists between layers.
 *   keep_new  uint8 [B, N]: the new layer's mask over the ORIGINAL positions,
 *             a subset of the previous layer's mask;
 *   dst_prev  int32 [B*N]: the previous layer's dst_idx (packed row of each
 *             original position, -1 where it was pruned);
 *   qp_prev/kp_prev/vp_prev: the previous layer's packed [cap, H, d] rows.
 * Writes cu_seqlens, dst_idx and src_idx exactly as rra_pack(keep_new) does
 * (src_idx keeps ORIGINAL flat positions b*N+j, so one rra_unpack or scatter
 * after the last layer restores the padded layout), and copies row
 * dst_prev[b*N+j] of each previous buffer to the new packed row of every
 * position keep_new keeps.  A position keep_new keeps that dst_prev marks
 * pruned records RRA_DEVERR_INDEX_RANGE and its rows are not copied.  The
 * previous and new buffers must not overlap (RRA_ERR_INVALID_ARG).  One
 * launch, asynchronous on `stream`. */
RRA_API rra_status rra_repack(const uint8_t* keep_new, const int32_t* dst_prev, int B, int N, int H, int d,
                              rra_dtype in_dtype, const void* qp_prev, const void* kp_prev,
                              const void* vp_prev, int32_t* cu_seqlens, int32_t* dst_idx,
                              int32_t* src_idx, void* qp, void* kp, void* vp, void* stream);

/* The index pass of rra_pack / rra_repack alone, for attention that reads
 * its rows in place (rra_attend_rows) instead of from a packed copy.
 *   keep      uint8 [B, N]: the layer's mask over the ORIGINAL positions;
 *   dst_prev  NULL (first layer), or the previous layer's dst_idx [B*N]
 *             (keep must then be a subset of the previous layer's mask);
 *   rows      NULL, or int32 [B*N]: rows[t] for every packed row t < T =
 *             cu_seqlens[B] is the row holding that token's data in the
 *             layer's input: src_idx[t] (the flat position, padded input)
 *             without dst_prev, dst_prev[src_idx[t]] (the row in the
 *             previous layer's packed buffers) with it.
 * Writes cu_seqlens, dst_idx and src_idx exactly as rra_pack(keep) does; no
 * row is copied.  A kept position that dst_prev marks pruned records
 * RRA_DEVERR_INDEX_RANGE and gets rows[t] = -1.  dst_prev must not be dst_idx
 * (RRA_ERR_INVALID_ARG).  One launch, asynchronous on `stream`. */
RRA_API rra_status rra_pack_index(const uint8_t* keep, const int32_t* dst_prev, int B, int N,
                                  int32_t* cu_seqlens, int32_t* dst_idx, int32_t* src_idx, int32_t* rows,
                                  void* stream);

/* Packed linear layer: the rest of a ViT block (QKV projection, output
 * projection, MLP) on the compact buffer, so pruned tokens cost no multiplies
 * there either (article, problem section: padding wastes bandwidth and
 * masked work).  c[t, :] = a[t, :] W^T (+ bias) for t < T = cu_seqlens[B],
 * T read on the device; rows t >= T of c are not written.
 *   a    [cap, K] of in_dtype (F16 or BF16), the packed rows;
 *   w    [N, K] of in_dtype (the nn.Linear weight layout);
 *   bias float [N] or NULL (16-byte aligned);
 *   c    [cap, N] of out_dtype (F16, BF16 or F32).
 * K a multiple of 64, N a multiple of 128 (else RRA_ERR_UNSUPPORTED); fp32
 * accumulation (tcgen05, TMEM).  One launch; a cu_seqlens[B] outside
 * [0, cap] records RRA_DEVERR_INDEX_RANGE and writes nothing. */
RRA_API rra_status rra_linear_packed(const void* a, const void* w, const float* bias, const int32_t* cu_seqlens,
                                     int B, int cap, int K, int N, rra_dtype in_dtype, void* c,
                                     rra_dtype out_dtype, void* stream);

/* The step before the path, on the device (an EViT-like pruner; the
 * abstract names EViT among the pruners the pipeline serves but does not
 * spell out its rule).  Reading: an image's class token is its first kept
 * token; a kept token's score is the class token's softmax attention weight
 * on it (scale * <q_cls, k_j> over the image's kept tokens), averaged over
 * the heads.
 *   rra_cls_scores: packed q/k [cap, H, d] with cu_seqlens and src_idx (as
 *   rra_pack writes them) -> scores float [B, N] at the original positions,
 *   0 where no token is kept.  fp32 arithmetic.  One launch.
 *   rra_topk_keep: keep_new [B, N] = each image's first kept token of
 *   keep_prev plus the top ceil(m * keep_num / keep_den) of its m other
 *   kept tokens by score; equal scores go to the lower position, a NaN score
 *   counts as -inf.  0 <= keep_num <= keep_den, keep_prev and keep_new must
 *   not overlap (else RRA_ERR_INVALID_ARG).  One launch; O(N^2) comparisons
 *   per image (N <= 1024). */
RRA_API rra_status rra_cls_scores(const void* qp, const void* kp, const int32_t* cu_seqlens,
                                  const int32_t* src_idx, int B, int N, int H, int d, float scale,
                                  rra_dtype in_dtype, float* scores, void* stream);
RRA_API rra_status rra_topk_keep(const float* scores, const uint8_t* keep_prev, int B, int N, int keep_num,
                                 int keep_den, uint8_t* keep_new, void* stream);

/* Bidirectional ragged attention on packed buffers (method overview,
 * bullet 2; abstract).  For image b with rows s = cu[b] .. e = cu[b+1]-1 and
 * head h, for every row i in [s, e]:
 *   O[i, h, :] = sum_j softmax_j(scale * <Q[i,h,:], K[j,h,:]>) V[j, h, :],
 *   j over [s, e] only (no causal mask).  One kernel launch; the grid is sized
 * from max_seqlen (an upper bound on every image's length) and lengths are
 * read on the device.
 * qp, kp and vp must span B*max_seqlen rows (the tile loads may read rows
 * up to that bound past the last image; what they hold is never used).
 *   src_idx == NULL: `o` is packed [cap, H, d] and row i is written at row i.
 *   src_idx != NULL: `o` is padded [B, N, H, d] and row i is written at flat
 *   position src_idx[i] (the unpack fused into the epilogue, bullet 3); rows
 *   at pruned positions are not touched (rra_pack's out_zero_fill sets them).
 * An image with zero rows writes nothing. */
RRA_API rra_status rra_attend(const void* qp, const void* kp, const void* vp,
                              const int32_t* cu_seqlens, int B, int max_seqlen, int H, int d,
                              float scale, rra_dtype in_dtype, void* o, rra_dtype out_dtype,
                              const int32_t* src_idx, int N, void* stream);

/* rra_attend, blocking until its output is complete, without a stream
 * synchronisation: the kernel's last CTA to finish publishes a ticket to a
 * page-locked host word (system-scope release after every CTA's stores),
 * and the calling thread polls that word.  Same arguments, layouts and
 * results as rra_attend.  Returns RRA_OK once o holds every row.  After
 * ~2 ms of polling the call falls back to cudaStreamSynchronize (long calls,
 * or a kernel that failed), so an asynchronous error still comes back as
 * RRA_ERR_CUDA.  Calls on one device are serialised by a lock (they share
 * the word and a device-side count).  The first call on a device allocates
 * that 64-byte page-locked host word (cudaHostAlloc, kept until the process
 * exits).  A call on a stream that is being captured returns
 * RRA_ERR_INVALID_ARG with nothing enqueued.  Made for host-side latency at serving
 * sizes (the abstract's dispatch-floor comparison): polling a coherent host
 * word returns sooner than a stream synchronisation does. */
RRA_API rra_status rra_attend_wait(const void* qp, const void* kp, const void* vp,
                                   const int32_t* cu_seqlens, int B, int max_seqlen, int H, int d,
                                   float scale, rra_dtype in_dtype, void* o, rra_dtype out_dtype,
                                   const int32_t* src_idx, int N, void* stream);

/* The same attention without a packed copy of the inputs: row t of image
 * b's sequence is read straight from the padded q/k/v [B, N, H, d] at flat
 * position src_idx[t] (TMA gather of 4 rows at a time) and the output row
 * is written to out [B, N, H, d] at the same position (rows at pruned
 * positions untouched).  cu_seqlens and src_idx are rra_pack's; every
 * image's length must be <= N.  This is rra_pipeline's attention step
 * (method overview, bullets 2-3, with the pack's row copy folded into the
 * attention's tile loads). */
RRA_API rra_status rra_attend_gather(const void* q, const void* k, const void* v,
                                     const int32_t* cu_seqlens, const int32_t* src_idx, int B, int N,
                                     int H, int d, float scale, rra_dtype in_dtype, void* out,
                                     rra_dtype out_dtype, void* stream);

/* rra_attend with the pack's row copy folded into the tile loads: the
 * sequence of image b is packed rows t = cu[b] .. cu[b+1]-1 as usual, but the
 * Q/K/V data of row t is read from row rows[t] of q/k/v [src_rows, H, d]
 * (TMA gather of 4 rows at a time), and the output is packed: o[t] for
 * t < T (o [cap, H, d], rows >= T untouched).  With rows from
 * rra_pack_index this is one layer of progressive pruning without a packed
 * copy: padded q/k/v (src_rows = B*N) at the first layer, the previous
 * layer's packed q/k/v at a pruning layer.  max_seqlen bounds every image's
 * length (longer images record RRA_DEVERR_SEQ_TOO_LONG and are skipped); a
 * row outside [0, src_rows) records RRA_DEVERR_INDEX_RANGE (its data read
 * as row 0's).  tcgen05 kernel only; one launch. */
RRA_API rra_status rra_attend_rows(const void* q, const void* k, const void* v, long long src_rows,
                                   const int32_t* rows, const int32_t* cu_seqlens, int B, int max_seqlen,
                                   int H, int d, float scale, rra_dtype in_dtype, void* o,
                                   rra_dtype out_dtype, float* cls, int cls_stride, void* stream);

/* rra_attend on packed buffers (src_idx NULL, packed output) that also
 * writes the class-token attention as a side output, for the pruning step
 * that follows a layer (EViT-like pruners rank tokens by the class token's
 * attention; abstract, both revisions):
 *   cls  float [B, H, cls_stride], 16-byte aligned: cls[b, h, i] for
 *        i < n_b = cu[b+1] - cu[b] is image b's class token's (its first
 *        row's) softmax weight, head h, on the image's row i, in fp32 from
 *        the same scores as the attention's; entries i >= n_b are
 *        unspecified, images with no rows leave theirs untouched.
 *   cls_stride  a multiple of 4, >= max_seqlen rounded up to a multiple of 16.
 * out_dtype must equal in_dtype (else RRA_ERR_UNSUPPORTED).  tcgen05 kernel
 * at every size; one launch.  rra_attend_rows takes the same two arguments
 * (cls NULL: no side output). */
RRA_API rra_status rra_attend_cls(const void* qp, const void* kp, const void* vp, const int32_t* cu_seqlens,
                                  int B, int max_seqlen, int H, int d, float scale, rra_dtype in_dtype, void* o,
                                  rra_dtype out_dtype, float* cls, int cls_stride, void* stream);

/* The pruning decision from that side output, one launch: image b's score
 * for its row i is the mean over the H heads of cls[b, h, i]; row 0 (the
 * class token) is kept with the top ceil((n_b-1) * keep_num / keep_den) of
 * rows 1 .. n_b-1 by score, exactly as rra_topk_keep ranks (equal scores to
 * the lower position, NaN as -inf).  keep_new [B, N] is written whole, at
 * the ORIGINAL positions src_idx[cu[b] + i] - b*N (rra_pack's src_idx);
 * scores, when not NULL, [B, N] receives each kept row's score there and 0
 * elsewhere (what rra_cls_scores would give).  cls_stride >= N.  An image
 * with n_b outside [0, N] records a device error and keeps nothing. */
RRA_API rra_status rra_topk_keep_cls(const float* cls, int cls_stride, const int32_t* cu_seqlens,
                                     const int32_t* src_idx, int B, int N, int H, int keep_num, int keep_den,
                                     uint8_t* keep_new, float* scores, void* stream);

/* The whole pruning step between two layers in one launch: the decision of
 * rra_topk_keep_cls from the side output of the layer before (cu_prev and
 * src_prev are that layer's indices) and the next layer's indices, exactly
 * as rra_pack_index(keep_new, dst_prev) would write them: cu_seqlens [B+1],
 * dst_idx [B*N], src_idx and rows [B*N] (rows[t]: the row of the previous
 * layer's packed buffers, cu_prev[b] + i, that holds the new row t -- the
 * input rra_attend_rows reads).  keep_new and scores may be NULL.  Image b's
 * new length is 1 + ceil((n_b-1) * keep_num / keep_den) (0 for n_b = 0), so
 * each image's new offset follows from cu_prev alone: every CTA sums the
 * lengths of the images before it, O(B) reads per image.  The new and
 * previous index buffers must not alias (RRA_ERR_INVALID_ARG). */
RRA_API rra_status rra_prune_index(const float* cls, int cls_stride, const int32_t* cu_prev,
                                   const int32_t* src_prev, int B, int N, int H, int keep_num, int keep_den,
                                   int32_t* cu_seqlens, int32_t* dst_idx, int32_t* src_idx, int32_t* rows,
                                   uint8_t* keep_new, float* scores, void* stream);

/* Unpack (method overview, bullet 3): out[b, j] = op[dst_idx[b*N+j]] when
 * dst_idx >= 0, else +0.  `op` is packed [cap, H, d] and `out` padded
 * [B, N, H, d], both of `dtype` (F16, BF16 or F32). */
RRA_API rra_status rra_unpack(const void* op, const int32_t* dst_idx, int B, int N, int H, int d,
                              rra_dtype dtype, void* out, void* stream);

/* The whole path, no host synchronisation, `out` [B, N, H, d] of out_dtype.
 * With a tcgen05 attention kernel (RRA_ATTEND_TCGEN05, _TCGEN05_LATENCY or
 * AUTO): ONE kernel launch that scans each image's keep row on the device,
 * gathers the kept Q/K/V rows straight from q/k/v (TMA gather4 in the
 * warp-specialised kernel, 16-byte cp.async copies in its small-grid form),
 * computes the attention and writes every output row -- kept positions get
 * the attention, pruned ones +0; the workspace is not touched.  With the
 * mma.sync kernel: rra_pack (with the row copy) then rra_attend on the
 * packed buffers, two launches; after the call the workspace holds
 * cu_seqlens, the pack indices and the packed Q/K/V.  `workspace` must hold
 * rra_workspace_bytes() bytes in either case. */
RRA_API rra_status rra_pipeline(const uint8_t* keep, const void* q, const void* k, const void* v,
                                int B, int N, int H, int d, float scale, rra_dtype in_dtype,
                                void* out, rra_dtype out_dtype,
                                void* workspace, size_t workspace_bytes, void* stream);

/* The same as rra_pipeline for inputs and output in pinned HOST memory:
 * enqueues host->device copies of keep/q/k/v into the caller's device
 * buffers (keep_d, q_d, k_d, v_d), the pipeline into out_d, and a
 * device->host copy of out_d into out_h, all on `stream`.  The caller syncs
 * the stream before reading out_h. */
RRA_API rra_status rra_pipeline_host(const uint8_t* keep_h, const void* q_h, const void* k_h,
                                     const void* v_h, int B, int N, int H, int d, float scale,
                                     rra_dtype in_dtype, void* out_h, rra_dtype out_dtype,
                                     uint8_t* keep_d, void* q_d, void* k_d, void* v_d, void* out_d,
                                     void* workspace, size_t workspace_bytes, void* stream);

/* The pipeline with inputs and output left in page-locked HOST memory and
 * no copies: the kernels read keep_h and the KEPT rows of q_h/k_h/v_h
 * straight from host memory over the CPU-GPU link, and write every row of
 * out_h (attention at kept positions, +0 at pruned ones) straight into host
 * memory.  Pruned input rows never cross the link, so the link carries
 * B*N + 3*T*H*d*size(in) bytes in and B*N*H*d*size(out) bytes out, T the
 * number of kept tokens.  With the tcgen05 kernel (RRA_ATTEND_TCGEN05 or
 * AUTO) and at most one (image, head, 128-query tile) unit per SM
 * (B*H*ceil(N/128) <= SM count, serving sizes): ONE launch of the fused
 * kernel, which copies the kept rows in with 16-byte cp.async copies (no
 * tensor maps over host memory) and writes every output row with plain
 * stores; the workspace is not touched.  Otherwise (larger batches, or the
 * mma.sync kernel selected): rra_pack (with the row copy) then the mma.sync
 * attention on the packed buffers in `workspace` (its epilogue writes whole
 * 128-byte lines, the efficient unit over the link), two launches.  Host
 * buffers: allocated by
 * cudaHostAlloc / cudaMallocHost or registered with cudaHostRegister, and
 * device-accessible (else RRA_ERR_INVALID_ARG, nothing enqueued); pageable
 * memory is refused.  `workspace`: DEVICE memory of rra_workspace_bytes()
 * bytes (else RRA_ERR_INVALID_ARG).  Asynchronous on `stream`: out_h is
 * complete once the stream has been synchronised. */
RRA_API rra_status rra_pipeline_mapped(const uint8_t* keep_h, const void* q_h, const void* k_h,
                                       const void* v_h, int B, int N, int H, int d, float scale,
                                       rra_dtype in_dtype, void* out_h, rra_dtype out_dtype,
                                       void* workspace, size_t workspace_bytes, void* stream);

/* Size of the scratch array rra_pipeline_static uses on each GPU (64 MiB). */
#define RRA_STATIC_SCRATCH_BYTES (64u * 1024u * 1024u)

/* rra_pipeline for callers that cannot allocate device memory.  The paper
 * has no counterpart to this entry point: it exists for code that may not
 * call cudaMalloc -- a plugin inside a host that owns all device memory, a
 * capture region it does not control, or a real-time loop that cannot
 * afford an allocation's implicit synchronisation -- and so cannot hand
 * rra_pipeline a workspace.  Same arguments and result as rra_pipeline
 * without the workspace: the scratch (cu_seqlens, pack indices, packed
 * Q/K/V) lives in one static device array of RRA_STATIC_SCRATCH_BYTES.
 *   - The array is taken on a device when the library's device code is
 *     loaded there: under CUDA's default lazy module loading that is the
 *     device's first rra_pipeline_static call (its address lookup below),
 *     under eager loading when the library is loaded.  It is held until the
 *     process exits.
 *   - Of the workloads the paper's configurations describe, tiny, serving
 *     (B <= 4) and batched B=64 (about 58 MB) fit; high-res B=32, N=577
 *     (about 85 MB) and the progressive B=256 layers (about 116 MB) do not.
 *   - Allocates nothing and calls no allocating routine.
 *   - Sizes whose workspace (rra_workspace_bytes) exceeds the array return
 *     RRA_ERR_UNSUPPORTED with nothing enqueued.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  The address is cached per device for the
 *     life of the process, like the rest of the library's per-device state
 *     (see rra_get_device_error): after cudaDeviceReset on a device, do not
 *     call this library on that device again in the same process.
 *   - All calls share the one array and it keeps the last call's contents
 *     (nothing in it has to start at zero).  Calls whose work overlaps on
 *     the GPU -- different streams without ordering between them -- race on
 *     it; order them on one stream or with events. */
RRA_API rra_status rra_pipeline_static(const uint8_t* keep, const void* q, const void* k, const void* v,
                                       int B, int N, int H, int d, float scale, rra_dtype in_dtype,
                                       void* out, rra_dtype out_dtype, void* stream);

/* A captured CUDA graph of one rra_pipeline call on fixed buffers: the
 * host-dispatch fix (problem section of the article).  rra_plan_create
 * validates the arguments exactly like rra_pipeline, runs the pipeline once
 * eagerly and captures it on a private stream; rra_plan_launch replays it on
 * `stream` with one graph launch.  The plan keeps the pointers, not the
 * data: later launches read whatever the buffers hold then. */
typedef struct rra_plan rra_plan;
RRA_API rra_status rra_plan_create(const uint8_t* keep, const void* q, const void* k, const void* v,
                                   int B, int N, int H, int d, float scale, rra_dtype in_dtype,
                                   void* out, rra_dtype out_dtype,
                                   void* workspace, size_t workspace_bytes, rra_plan** plan);
RRA_API rra_status rra_plan_launch(rra_plan* plan, void* stream);
RRA_API void rra_plan_destroy(rra_plan* plan);

/* Which kernel rra_attend and rra_pipeline launch; process-wide, returns
 * the previous choice (or -1 for an unknown value).
 *   RRA_ATTEND_TCGEN05  TMA tile loads + tcgen05.mma with TMEM accumulators,
 *                       warp-specialised persistent CTAs; rra_pipeline
 *                       gathers rows from the padded inputs (no packed copy);
 *   RRA_ATTEND_MMA_SYNC warp-level mma.sync kernel on packed buffers;
 *                       rra_pipeline packs with the row copy first;
 *   RRA_ATTEND_TCGEN05_LATENCY  tcgen05.mma with TMEM accumulators, one CTA
 *                       of four warps per (image, head, query tile) doing
 *                       every step in turn (cp.async loads, no warp
 *                       specialisation): the shortest chain for grids of
 *                       about one unit per SM; max_seqlen (rra_pipeline: N)
 *                       up to 256, the TCGEN05 kernel beyond;
 *   RRA_ATTEND_AUTO     (default) with max_seqlen <= 256: rra_pipeline
 *                       takes TCGEN05_LATENCY while the grid (B * H *
 *                       ceil(max_seqlen / 128) units) is at most four per
 *                       SM, rra_attend MMA_SYNC (the shortest chain on
 *                       packed buffers) while it is at most two per SM;
 *                       TCGEN05 otherwise. */
typedef enum {
  RRA_ATTEND_TCGEN05 = 0,
  RRA_ATTEND_MMA_SYNC = 1,
  RRA_ATTEND_AUTO = 2,
  RRA_ATTEND_TCGEN05_LATENCY = 3
} rra_attend_kernel;
RRA_API int rra_set_attend_kernel(int kernel);

/* Reads (and with clear != 0 resets) the device-side error code of the
 * current device: the word every launch records into unless its host
 * thread has bound one of its own (rra_bind_error_word).  Synchronous:
 * call it after the stream has been synced.  The word's address is cached
 * per device for the life of the process, like the rest of the library's
 * per-device state: after cudaDeviceReset on a device, do not call this
 * library on that device again in the same process. */
RRA_API rra_status rra_get_device_error(int32_t* code, int clear);

/* Per-call device error state.  rra_bind_error_word binds, for the calling
 * host thread, a caller-owned int32 in device memory (4-byte aligned, else
 * RRA_ERR_MISALIGNED) as the error word of every kernel this thread
 * enqueues from then on; NULL restores the device's own word.  Each call
 * (or stream, or plan) can so own its errors: two pipelines enqueued on two
 * streams with different words never see each other's codes.  A plan
 * records into the word bound when rra_plan_create ran.  The caller zeroes
 * the word before use; the first code recorded wins (later ones are kept
 * out).  rra_read_error_word copies the word to *code (and with clear != 0
 * zeroes it), synchronously; it returns RRA_ERR_DEVICE when the code is
 * nonzero. */
RRA_API rra_status rra_bind_error_word(int32_t* word);
RRA_API rra_status rra_read_error_word(int32_t* word, int32_t* code, int clear);

/* Bound, in clock cycles, on any one on-chip wait of the tcgen05 attention
 * kernels (0, the initial value: about one second).  A wait that runs out
 * makes the CTA record RRA_DEVERR_WAIT_TIMEOUT, give its own copies and
 * products a short grace period, release its tensor memory and return, its
 * output incomplete; the device stays usable.  A test hook for that failure
 * path: process-wide, applies to launches enqueued after the call; returns
 * the previous value (-1, nothing changed, for a negative argument). */
RRA_API long long rra_set_wait_limit(long long cycles);

/* Host-timed latency of rra_attend: `warmup` then `reps` repetitions of
 * {t0 = steady_clock; rra_attend(...); cudaStreamSynchronize; t1}; the
 * per-call microseconds go to samples_us[reps].  A measurement helper for
 * the dispatch-floor numbers of the abstract; it launches rra_attend only. */
RRA_API rra_status rra_time_attend_host(const void* qp, const void* kp, const void* vp,
                                        const int32_t* cu_seqlens, int B, int max_seqlen, int H,
                                        int d, float scale, rra_dtype in_dtype, void* o,
                                        rra_dtype out_dtype, const int32_t* src_idx, int N,
                                        void* stream, int warmup, int reps, double* samples_us);

/* Same helper for rra_attend_wait: {t0; rra_attend_wait(...); t1} (the call
 * returns once the output is complete, so no stream sync is added). */
RRA_API rra_status rra_time_attend_wait_host(const void* qp, const void* kp, const void* vp,
                                             const int32_t* cu_seqlens, int B, int max_seqlen, int H,
                                             int d, float scale, rra_dtype in_dtype, void* o,
                                             rra_dtype out_dtype, const int32_t* src_idx, int N,
                                             void* stream, int warmup, int reps, double* samples_us);

/* Same helper for a graph plan: {t0; rra_plan_launch; sync; t1}. */
RRA_API rra_status rra_time_plan_host(rra_plan* plan, void* stream, int warmup, int reps,
                                      double* samples_us);

/* Reference floor for the two helpers above: {t0; launch an empty kernel;
 * sync; t1}.  It measures this host + driver + GPU's own dispatch floor, the
 * quantity the abstract compares across attention implementations. */
RRA_API rra_status rra_time_null_host(void* stream, int warmup, int reps, double* samples_us);

RRA_API const char* rra_status_string(rra_status status);
RRA_API const char* rra_last_error_message(void);

/* Number of this library's kernel launches enqueued by this process so far
 * (every entry point adds the launches it makes; graph replays through
 * rra_plan_launch add the launches the graph holds). */
RRA_API uint64_t rra_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* RRA_H */
