/*
 * pck.h -- C ABI of libpck: attention of query rows over a resident shared-prefix KV cache
 * on one GB300 (sm_103a).
 *
 * The calls follow the problem statement of the ATTEND.PREFIX.* wire forms on the page
 * "ATTEND.* and ATTEND.PREFIX.*", section "Wire forms" (STORE / LOOKUP / QUERY /
 * QUERY_FUSED / QUERY_SPARSE_AUTO / QUERY_SPARSE_AUTO_FUSED), with explicit M, dtypes and
 * pointer ownership. The mlx4g32 tier follows "Shared KV Cache Serving -- Pion as LLM
 * Memory", section "Quantized tier -- mlx4g32".
 *
 * Conventions for every call:
 *  - Tensor pointers (Q, O, LSE, K, V, K_suf, V_suf, records, idx_out) are DEVICE pointers
 *    on the context's device, caller-owned, contiguous, and must stay valid until the stream
 *    reaches the call. O, K, V and Q must be 16-byte aligned, and K_suf / V_suf too when M > 1
 *    (PCK_EINVAL otherwise). head_map is a small HOST array (int32[H_q], entries in [0, H_kv));
 *    NULL means the grouped default h / (H_q / H_kv).
 *  - `stream` is a cudaStream_t passed as void*; NULL is the legacy default stream.
 *  - Calls are asynchronous on `stream`. Argument, shape and slot errors are detected on the
 *    host and returned before anything is launched. Asynchronous CUDA errors are reported as
 *    PCK_ECUDA by pck_sync or by a later call.
 *  - One context serialises its work: queries on one context must be issued on one stream
 *    (they share the context's split-K workspace). Use one context per stream otherwise.
 *  - Scores are tau * q.k with tau = 1/sqrt(D). LSE is in natural-log units of the scaled
 *    logits: LSE = ln(sum_t exp(tau q.k_t)). O is fp32 [H_q, M, D], LSE fp32 [H_q, M].
 *  - On a non-OK status, pck_last_error(ctx) holds a one-line reason.
 */
#ifndef PCK_H
#define PCK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. PCK_MISS matches the wire's +MISS / "-ERR session not found"; PCK_COLDMISS
 * matches STATUS_COLDMISS = 0x03 of the binary lane ("Shared KV Cache Serving", section
 * "Cold-tier state machine"): the slot was evicted by LRU and must be stored again. */
#define PCK_OK            0
#define PCK_MISS          1
#define PCK_COLDMISS      3
#define PCK_EINVAL       (-1)
#define PCK_EUNSUPPORTED (-2)
#define PCK_ENOMEM       (-3)
#define PCK_ECUDA        (-4)

/* Resident formats of a slot. */
#define PCK_FMT_FP16     0  /* fp16 K/V */
#define PCK_FMT_MLX4G32  1  /* int4, group 32, affine, fp16 scale + fp16 bias per group */

/* Element types of caller tensors. */
#define PCK_DT_F32       0
#define PCK_DT_F16       1

/* Head dimensions with kernels: fp16 slots 32, 64, 96, 128, 160, 192, 256 (M = 1 and M > 1) and
 * 512 (M = 1 only: M > 1 returns PCK_EUNSUPPORTED); mlx4g32 slots 64, 128, 192, 256 (M > 1: 64,
 * 128); QUERY_SPARSE_AUTO(_FUSED) 64, 128, 256; QUERY_SPARSE every fp16 slot. More than 8 q heads
 * per kv head (4 at D = 512) are split into work groups, each of which reads the kv head. */
#define PCK_MAX_BATCH    64   /* descriptors per pck_query_batch call */
#define PCK_MAX_HEADS    64   /* H_q and H_kv limit */

typedef struct pck_ctx pck_ctx;

typedef struct pck_info_t {
    int64_t slots_used;       /* resident (sid, layer) slots */
    int64_t slots_max;        /* capacity (LRU eviction beyond it) */
    int64_t cold_entries;     /* evicted keys remembered for PCK_COLDMISS */
    int64_t bytes_resident;   /* device bytes held by resident K/V (+ block means) */
    int64_t queries_served;   /* query calls that launched work */
    int64_t stores;           /* store calls that launched work */
    int64_t evictions;        /* LRU demotions */
} pck_info_t;

/* One M=1 query of a pck_query_batch call. */
typedef struct pck_query_desc {
    const char *sid;          /* session id (NUL-terminated) */
    int layer;
    const void *Q;            /* device [H_q, D], q_dtype of the batch */
    float *O;                 /* device [H_q, D] fp32 */
    float *LSE;               /* device [H_q] fp32, or NULL */
    const void *K_suf;        /* device fp16 [H_kv, S_suf, D], or NULL when S_suf == 0 */
    const void *V_suf;
} pck_query_desc;

/* One M=1 query of a pck_query_sparse_batch call. */
typedef struct pck_sparse_desc {
    const char *sid;          /* session id (NUL-terminated) */
    int layer;
    const void *Q;            /* device [H_q, D], q_dtype of the batch */
    float *O;                 /* device [H_q, D] fp32 */
    float *LSE;               /* device [H_q] fp32, or NULL */
    const void *K_suf;        /* device fp16 [H_kv, S_suf, D], or NULL when S_suf == 0 */
    const void *V_suf;
    int32_t *idx_out;         /* device [H_q, min(K_top, nb)] selected blocks (ascending), or NULL */
} pck_sparse_desc;

/* Create a context on CUDA device `device` with room for `max_slots` resident (sid, layer)
 * slots (<= 0 selects 256, the per-worker slot table size of the pages' session cache).
 * Allocates the split-K workspace. Returns PCK_OK and *out, or PCK_ECUDA / PCK_ENOMEM. */
int pck_create(pck_ctx **out, int device, int max_slots);

/* Free every resident slot and the workspace. Synchronises the device first. NULL is a no-op. */
void pck_destroy(pck_ctx *ctx);

/* One-line description of the last error on ctx ("" if none). Owned by ctx. */
const char *pck_last_error(const pck_ctx *ctx);

/* ATTEND.PREFIX.STORE <sid> <layer> <H> <N> <D> <K_blob> <V_blob>.
 * K, V: device [H_kv, N, D], src_dtype F16 or F32. fmt FP16 keeps fp16 K/V resident;
 * fmt MLX4G32 quantises both on the device (same arithmetic as pck_quantize_mlx4g32) and keeps
 * the codes/scales/biases resident. Replaces an existing slot with the same key. The library
 * copies K/V into its own memory: the caller may reuse K/V once the stream passes the call.
 * D: see above; H_kv <= 64, N >= 1. Errors: EINVAL, EUNSUPPORTED, ENOMEM. */
int pck_store(pck_ctx *ctx, const char *sid, int layer, int H_kv, int N, int D, int fmt,
              const void *K, const void *V, int src_dtype, void *stream);

/* Store pre-quantised mlx4g32 records (token-major [N, rec] with rec = H_kv*D/8*4 + 2*(H_kv*D/32)*2
 * bytes: codes words, then scales, then biases; see pck_quantize_mlx4g32) as a MLX4G32 slot. */
int pck_store_records(pck_ctx *ctx, const char *sid, int layer, int H_kv, int N, int D,
                      const void *K_rec, const void *V_rec, void *stream);

/* ATTEND.PREFIX.LOOKUP: PCK_OK if (sid, layer) is resident, PCK_COLDMISS if it was evicted,
 * PCK_MISS otherwise. */
int pck_lookup(pck_ctx *ctx, const char *sid, int layer);

/* Drop (sid, layer), or every layer of sid when layer < 0. Memory is released in stream order
 * on `stream` (queued work on that stream still sees valid K/V). Returns the number dropped. */
int pck_drop(pck_ctx *ctx, const char *sid, int layer, void *stream);

/* Precompute the block means of K (fp32, [H_kv, ceil(N/B), D]) used by the sparse selector, and
 * (at D in {64, 128, 256} with at most 1024 blocks) their fp16 hi + lo copy for the one-kernel form.
 * The sparse queries build them on first use per (slot, B); this lets a caller do it at store
 * time (e.g. before capturing a CUDA graph). Only fp16 slots. The means of all slots share
 * device memory the context sets aside in large chunks (packed together, the batched sparse
 * form reads them faster); a build that would allocate while `stream` is being captured
 * returns PCK_EINVAL, so a captured sparse call needs its slots' means built beforehand. */
int pck_build_block_means(pck_ctx *ctx, const char *sid, int layer, int B, void *stream);

/* ATTEND.PREFIX.QUERY <sid> <layer> <H> <D> <top_k> <Q_blob> [<fa_window>].
 * Q: device [H_q, M, D] of q_dtype. M == 1: split-K decode over the slot (fp16 or mlx4g32).
 * M > 1: tiled tensor-core kernel; needs q_dtype F16 (PCK_EUNSUPPORTED otherwise). Over an
 * mlx4g32 slot (D in {64, 128}) the call first dequantises the slot into a stream-ordered
 * temporary of H_kv * N * 8 * D bytes, each value as an fp16 hi + lo pair, and attends to it
 * with the same kernel at width 2D, so K and V keep ~22 bits.
 * top_k: 0 or >= N (dense); smaller values are PCK_EUNSUPPORTED.
 * fa_window (listed on every QUERY form of the pages, never defined there; this library's reading):
 * 0 = no window; W > 0 = a sliding attention window: query row i, at absolute position
 * p_i = N + S_suf - M + i (prefix positions 0 .. N-1, then the suffix), sees only positions
 * p_i - W + 1 .. p_i (and, with causal, no suffix key past its own). Built for every dense QUERY
 * form (M = 1 and M > 1, both formats, with or without a suffix); the sparse forms take W = 0
 * only (PCK_EUNSUPPORTED otherwise); W < 0 is PCK_EINVAL.
 * Writes O [H_q, M, D] and, if LSE != NULL, LSE [H_q, M]. */
int pck_query(pck_ctx *ctx, const char *sid, int layer, int H_q, int D, int M, int q_dtype,
              const void *Q, const int32_t *head_map, int top_k, int fa_window,
              float *O, float *LSE, void *stream);

/* ATTEND.PREFIX.QUERY_FUSED: prefix attention plus attention to a dense suffix
 * K_suf/V_suf (device fp16 [H_kv, S_suf, D]), merged by online softmax in the same launch.
 * causal != 0: query row i (of M) sees suffix keys j <= S_suf - M + i (bottom-right aligned);
 * causal == 0: every row sees the whole suffix. The merged LSE is written if LSE != NULL. */
int pck_query_fused(pck_ctx *ctx, const char *sid, int layer, int H_q, int D, int M, int S_suf,
                    int H_kv, int q_dtype, const void *Q, const void *K_suf, const void *V_suf,
                    const int32_t *head_map, int causal, int fa_window,
                    float *O, float *LSE, void *stream);

/* ATTEND.PREFIX.QUERY_SPARSE_AUTO: M=1. Scores the slot's B-token blocks by
 * tau * q_h . mean(K of the block), keeps the K_top best per q head (ties -> lower index,
 * K_top clamped to ceil(N/B)), and attends only to their tokens. idx_out (device
 * int32 [H_q, min(K_top, nblocks)], nullable) receives the selected blocks, sorted ascending.
 * fp16 slots only. */
int pck_query_sparse_auto(pck_ctx *ctx, const char *sid, int layer, int H_q, int D, int B,
                          int K_top, int H_kv, int q_dtype, const void *Q,
                          const int32_t *head_map, int fa_window,
                          float *O, float *LSE, int32_t *idx_out, void *stream);

/* ATTEND.PREFIX.QUERY_SPARSE_AUTO_FUSED: the sparse prefix plus a dense suffix (device fp16
 * [H_kv, S_suf, D]) merged by online softmax. */
int pck_query_sparse_auto_fused(pck_ctx *ctx, const char *sid, int layer, int H_q, int D, int B,
                                int K_top, int H_kv, int S_suf, int q_dtype, const void *Q,
                                const void *K_suf, const void *V_suf, const int32_t *head_map,
                                int fa_window, float *O, float *LSE, int32_t *idx_out,
                                void *stream);

/* ATTEND.PREFIX.QUERY_SPARSE <sid> <layer> <H> <D> <K_sparse_max> <Q> <indices> <counts>
 * ("ATTEND.* and ATTEND.PREFIX.*", command table: M=1 attention restricted to caller-supplied
 * per-head token indices, e.g. from a learned router). Q: device [H_q, D] of q_dtype; O: device
 * fp32 [H_q, D]; LSE: device fp32 [H_q] or NULL. indices: HOST int32 [H_q, K_sparse_max], row h
 * holding counts[h] prefix token positions (HOST int32 [H_q]) that q head h attends to, of kv
 * head head_map[h] (NULL head_map: h / (H_q / H_kv)). Checked on the host before anything is
 * launched: 1 <= counts[h] <= K_sparse_max, positions in [0, N) and strictly ascending (no
 * duplicates), else PCK_EINVAL. fp16 slots, H_q <= 64, fa_window 0. The index lists are copied
 * to the device with a pageable host-to-device copy (the host arrays may be reused once the call
 * returns; the call cannot be captured in a CUDA graph); the selected tokens are gathered into a
 * stream-ordered temporary and attended by the split-K decode. */
int pck_query_sparse(pck_ctx *ctx, const char *sid, int layer, int H_q, int D, int K_sparse_max, int q_dtype,
                     const void *Q, const int32_t *indices, const int32_t *counts, const int32_t *head_map,
                     int fa_window, float *O, float *LSE, void *stream);

/* Copy the slot's block means (fp32 [H_kv, ceil(N/B), D], built first when absent; see
 * pck_build_block_means) into the device buffer `out`. */
int pck_get_block_means(pck_ctx *ctx, const char *sid, int layer, int B, float *out, void *stream);

/* n independent M=1 queries of one shape (H_q, H_kv, D, S_suf, q_dtype, head_map) in ONE
 * launch: the whole batch is split evenly over the GPU. 1 <= n <= PCK_MAX_BATCH. All slots
 * must have the same format. */
int pck_query_batch(pck_ctx *ctx, int n, const pck_query_desc *descs, int H_q, int H_kv, int D,
                    int S_suf, int q_dtype, const int32_t *head_map, void *stream);

/* pck_query_batch over HOST buffers: descs[i].Q, K_suf, V_suf (inputs) and O, LSE (outputs) are
 * page-locked host pointers (cudaHostAlloc, cudaHostRegister or a pinned tensor), 16-byte
 * aligned; everything else is as pck_query_batch. The call moves the bytes itself, on `stream`:
 * a copy kernel reads the inputs over the host link into the context's staging memory (at most
 * PCK_HOST_STAGE_BYTES per call), the batch runs on the staged copies, and its merge kernel
 * writes O and LSE straight into the host buffers. The outputs are valid, and the inputs may be
 * reused, once `stream` has been synchronised. Errors: as pck_query_batch; PCK_EINVAL for a
 * pointer that is not page-locked host memory; PCK_EUNSUPPORTED above the staging size. */
#define PCK_HOST_STAGE_BYTES (16u << 20)
int pck_query_batch_host(pck_ctx *ctx, int n, const pck_query_desc *descs, int H_q, int H_kv, int D,
                         int S_suf, int q_dtype, const int32_t *head_map, void *stream);

/* n independent ATTEND.PREFIX.QUERY_SPARSE_AUTO(_FUSED) queries (page "ATTEND.* and
 * ATTEND.PREFIX.*", section "Wire forms"; batching them is this library's addition, as for
 * pck_query_batch) of one shape (H_q, H_kv, D, B, K_top, S_suf, q_dtype, head_map) over fp16
 * slots of the same N. A batch of at least 32 work items (query x group of up to 8 q heads of a
 * kv head, 4 at D = 256) over at most 1024 blocks per kv head, with 16-byte aligned suffixes,
 * runs as ONE kernel with a CTA per work item (scores, top-K, union, gather decode of the union
 * and the suffix, merge); otherwise the block scores of all queries run in one scoring launch,
 * their top-K selections in one selection launch, and their gathers (+ suffixes) in one split-K
 * decode and its merge (four launches). Each query is as pck_query_sparse_auto_fused
 * (S_suf > 0) or pck_query_sparse_auto (S_suf == 0) would compute it alone. The first sparse
 * call on a slot builds its block means (and their fp16 hi + lo copy, which the one-kernel form
 * scores from) with stream-ordered allocations: call pck_build_block_means, or make a first
 * call, before capturing the call in a CUDA graph.
 * 1 <= n <= PCK_MAX_BATCH. Errors: EINVAL, EUNSUPPORTED (slots of different N, B not a multiple
 * of 16, K_top > 64, fa_window), MISS / COLDMISS for an absent slot. */
int pck_query_sparse_batch(pck_ctx *ctx, int n, const pck_sparse_desc *descs, int H_q, int H_kv, int D,
                           int B, int K_top, int S_suf, int q_dtype, const int32_t *head_map,
                           void *stream);

/* mlx4g32 quantiser (store side). X: device [rows, kv_dim] of src_dtype (F16 or F32);
 * out_records: device [rows, rec] bytes, rec = kv_dim/2 + kv_dim/8. Per group of 32:
 * mn/mx as fp32, s32 = (mx - mn)/15 in fp32, scale = fp16(s32) (rounded BEFORE the codes are
 * chosen), bias = fp16(mn), code = clamp(rint((x - bias)/scale), 0, 15) in fp32, all codes 0 when
 * scale == 0; code j fills bits 4*(j%8) .. 4*(j%8)+3 of word j/8. kv_dim % 32 == 0. Inputs must be
 * finite and within the fp16 range. Needs no context. */
int pck_quantize_mlx4g32(const void *X, int src_dtype, int64_t rows, int kv_dim,
                         void *out_records, void *stream);

/* The KV.PREFIX.WARM / V.FETCH RANGE form of stored mlx4g32 records ("Shared KV Cache Serving
 * -- Pion as LLM Memory", sections "KV.PREFIX.WARM" and "Cold-tier state machine"; "V.* -- the
 * V-store", V.FETCH): records (device, token-major [N, rec] as in pck_store_records, 4-byte
 * aligned) -> out (device, [H_kv, N, D], 16-byte aligned), the dequantised x = scale * code +
 * bias rounded once to fp32 (out_dtype F32), or that fp32 value rounded to fp16 (F16): the
 * dequantise and the [N, H*D] -> [H, N, D] transpose in one pass. H_kv * D % 32 == 0,
 * D % 8 == 0. Needs no context. Errors: EINVAL, ECUDA. */
int pck_dequantize_mlx4g32(const void *records, int64_t N, int H_kv, int D, int out_dtype, void *out,
                           void *stream);

/* Attention of M=1 queries over mlx4g32 records the caller holds, allocating nothing.
 * The pages have no counterpart: it exists for callers that cannot allocate device memory at
 * call time (code running under another framework's allocator budget, a request path that must
 * not touch the allocator, or a process without a pck context). It runs the same kernels as
 * pck_store_records + pck_query_fused (M=1), with the same split of the work, but all scratch
 * lives in device arrays compiled into libpck (PCK_NOALLOC_SCRATCH_BYTES per GPU, held from
 * library load until process exit).
 * K_rec, V_rec: device token-major records [N, rec] as in pck_store_records. Q: device [H_q, D];
 * O: device fp32 [H_q, D]; LSE: device fp32 [H_q] or NULL; K_suf/V_suf: device fp16
 * [H_kv, S_suf, D] or NULL when S_suf == 0. Limits: H_kv * ceil(N/16) * 20*D bytes of resident
 * tiles <= 16 MiB, D in {64, 128, 192, 256}; larger inputs return PCK_EUNSUPPORTED before any
 * launch. The first call on a device (or the first pck_noalloc_status there) looks up the
 * scratch addresses and the kernels' occupancy: make it before any stream capture. All calls
 * share the scratch: calls that overlap on the GPU (other streams or host threads) race and
 * must be serialised by the caller. Returns PCK_OK, PCK_EINVAL, PCK_EUNSUPPORTED or PCK_ECUDA
 * (no context, so no pck_last_error text). A kernel-side failure (see pck_sync's codes) shows
 * only in pck_noalloc_status. */
#define PCK_NOALLOC_SCRATCH_BYTES ((16u << 20) + (16u << 20) + 64u * 4u)
int pck_attend_records_noalloc(int H_kv, int N, int D, const void *K_rec, const void *V_rec, int H_q,
                               int q_dtype, const void *Q, const int32_t *head_map, int S_suf,
                               const void *K_suf, const void *V_suf, float *O, float *LSE, void *stream);

/* Status of the pck_attend_records_noalloc calls made on the current device since the last
 * status call. Synchronises `stream`, reads the scratch's device error word and clears it.
 * PCK_OK: no kernel reported an error. PCK_ECUDA: a CUDA error, or some call's kernels set a
 * device error code (written to *code when code != NULL; the codes are pck_sync's): at least
 * one of those calls wrote invalid results. Callers that use the results should check it. */
int pck_noalloc_status(void *stream, int *code);

/* Counters of ctx. */
int pck_info(pck_ctx *ctx, pck_info_t *out);

/* Synchronise `stream` and report any asynchronous CUDA error as PCK_ECUDA. Also PCK_ECUDA when
 * a kernel's bounded wait gave up since the last check (a TMA stage or pipeline barrier that
 * never completed). The kernel then skipped the rest of its work, so the affected results are
 * invalid. pck_last_error names the code: 1 decode ring stage, 2 prefill producer, 3 prefill
 * MMA warp, 4 prefill softmax, 5 prefill final O, 6 sparse scoring copy, 7 an fp32 Q element
 * of an M=1 query with |q| * log2(e) / sqrt(D) >= 65504 (or not finite): the M=1 kernels
 * carry q * log2(e) / sqrt(D) as an fp16 hi + lo pair, so |q| < 65504 * sqrt(D) / log2(e)
 * (e.g. 363,000 at D = 64) is the valid range. The error word and the selector's counters
 * are then reset, so the context stays usable. */
int pck_sync(pck_ctx *ctx, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PCK_H */
