// pck_kernels.h -- host-side declarations of the kernel launchers (internal to libpck).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "pck_common.cuh"

namespace pck {

constexpr int PCK_MAXH = 64;

// store side
cudaError_t launch_quantize(const void* X, int src_f16, int64_t rows, int kv_dim, void* out, cudaStream_t st, int sms);
// DS: head dimension of the written layout (0 = D; DS > D pads every row with zero columns);
// release: 1 lets the next kernel start before this one ends (only for a reader that waits for it)
cudaError_t launch_relayout_fp16(const void* K, const void* V, int src_f16, int H_kv, int N, int D, int ntiles,
                                 void* out, cudaStream_t st, int sms, int DS = 0, int release = 0);
cudaError_t launch_relayout_mlx4(const void* Krec, const void* Vrec, int head_rows, int H_kv, int N, int D, int ntiles,
                                 void* out, cudaStream_t st, int sms);
// QUERY_SPARSE: the tokens idx[h][0 .. counts[h]) of kv head head_map[h] of a resident fp16 slot,
// gathered into one compact fp16 slot per q head h (at out + h * head_stride)
cudaError_t launch_gather_fp16(const void* tiles, int ntiles, int D, const int* idx, const int* counts,
                               const int8_t* head_map, int H_q, int kmax, size_t head_stride, void* out, cudaStream_t st);
// mlx4g32 slot tiles -> an fp16 slot of head dimension 2D holding [hi | lo] fp16 pairs of the values
cudaError_t launch_mlx4_split(const void* tiles, int H_kv, int ntiles, int D, void* out, cudaStream_t st);
// token-major records [N, H_kv*D] -> [H_kv, N, D] fp32 or fp16
cudaError_t launch_dequant_records(const void* rec, int64_t N, int H_kv, int D, int out_f16, void* out, cudaStream_t st,
                                   int sms);

// M=1 split-K decode (dense or sparse item sequences), fused suffix and merge
struct DecodeLaunchInfo {
    int stage_bytes;
    int nstage;
    int smem_bytes;
    int ctas_per_sm;
};
DecodeLaunchInfo decode_launch_info(int fmt, int D, int ncb);
// the M=1 kernels' head dimensions: 32, 64, 96, 128, 160, 192, 256 for fp16 slots; 64, 128, 192,
// 256 for mlx4g32 slots
bool decode_dim_ok(int fmt, int D);
DecodeLaunchInfo decode_launch_info_xd(int fmt, int D, int ncb);   // D in {32, 96, 160, 192}
cudaError_t launch_decode_xd(int fmt, int D, const DecodeParams& p, int n_ctas, cudaStream_t st);
// How one decode launch splits its work. Dense: `total` units (16-token tiles) over items of at
// most `vmax` units each are cut into ranges of tpw units, one per prefix worker (a warp), with
// at least max(ceil(vmax / 64), 4) units per range (an item has at most ~64 pieces to merge, and
// a piece is worth its start-up), and at most one wave of resident warps (ctas_per_sm CTAs of
// DECODE_WARPS warps on each of `sms` SMs) together with the items' suffix warps. Sparse: `total` bounds the units, and every resident
// prefix warp takes a share on the device. The partial slots the launch writes (one per prefix
// worker, per item, and per suffix piece) must fit `max_slots`; ranges grow until they do.
struct DecodePlan {
    int tpw;              // dense: units per prefix worker
    int n_workers;        // prefix workers
    int n_suf;            // suffix pieces per item (ceil(S_suf / 16))
    int n_ctas;           // CTAs of the launch
    int64_t slots;        // partial slots written
};
// false when the launch cannot fit (the item and suffix slots alone exceed max_slots).
// Dense launches (p->sparse == 0) cut every item into whole pieces of about tpw tiles (p->ppi,
// p->wbase; one worker per piece, so that no worker's range straddles two items: a worker that
// starts a second item finishes late) unless whole pieces would be over 5 % longer than the plain
// split (items long against the warps' share), where p->aligned stays 0 and ranges of tpw tiles
// run across item boundaries. p's descriptors, n_desc and n_groups must be set.
bool plan_decode(DecodeParams* p, int64_t total, int vmax, int n_items, int S_suf, int sms, int ctas_per_sm,
                 int64_t max_slots, DecodePlan* out);
int decode_ncb(const DecodeParams& p);   // 4-head column blocks the mlx4g32 kernel needs for p
cudaError_t launch_decode(int fmt, int D, const DecodeParams& p, int n_ctas, cudaStream_t st);

// sparse selector
cudaError_t launch_block_means(const void* tiles, int H_kv, int N, int D, int ntiles, int B, float* kmean,
                               cudaStream_t st, int sms);
// One session of a selector launch (a query against one slot).
struct SelSession {
    const float* kmean;      // [H_kv, nb, D]
    const void* Q;           // [H_q, D]
    float* scores;           // workspace [H_q, nb]
    int* idx_out;            // [H_q, K_eff] or nullptr
    int* sel_blocks;         // [n_groups, sel_max]
    uint8_t* sel_mask;       // [n_groups, sel_max]
};
// Block scoring + top-K selection for n_sess sessions of the same shapes (one launch each).
struct SelectParams {
    int q_f16;
    int H_q, H_kv, D, nb, K_top, K_eff, sel_max, n_groups, n_sess;
    int tpb;                 // 16-token tiles per block (B / 16)
    int ntiles;              // tiles of the slots (ceil(N / 16))
    float tau;
    int* item_cnt;           // [n_sess * n_groups] selected tiles of each (session, group) item
    int* item_base;          // [n_sess * n_groups + 1] exclusive prefix of item_cnt (the decode's units)
    unsigned* done;          // items selected so far (the last one writes item_base and resets it)
    int* err;                // device error word
    int8_t head_map[PCK_MAXH];
    WorkGroup grp[MAX_GROUPS];
    SelSession sess[MAX_DESC];
};
cudaError_t launch_select(const SelectParams& p, cudaStream_t st, int sms);

// The whole block-mean sparse query in one kernel (one CTA per (session, work group)): scores,
// top-K and union in shared memory, gather decode of the union plus the dense suffix, and the
// merge of the CTA's pieces. Work groups hold at most sparse_fused_gmax(D) q heads.
// fp32 block means [H_kv, nb, D] -> fp16 hi + lo pairs (x = hi + lo to ~22 bits) in the resident
// K-tile layout with blocks as tokens: per kv head and group of 16 blocks, a hi part and a lo part
// of 32 D bytes each (core matrices [block group][d chunk]); blocks past nb are zero.
cudaError_t launch_block_means_split(const float* kmean, int H_kv, int nb, int D, uint8_t* out, cudaStream_t st);
struct FusedSession {
    const uint8_t* kmean;    // split block means (launch_block_means_split) of the slot
    const void* Q;           // [H_q, D]
    const uint8_t* kv;       // resident fp16 slot
    const __half* Ksuf;      // [H_kv, S_suf, D] or nullptr
    const __half* Vsuf;
    float* O;                // [H_q, D]
    float* LSE;              // [H_q] or nullptr
    int* idx_out;            // [H_q, K_eff] or nullptr
};
struct FusedSparseParams {
    FusedSession sess[MAX_DESC];
    WorkGroup grp[MAX_GROUPS];
    int n_sess, n_groups, H_q, D, N, ntiles, nb, tpb, K_eff, S_suf, q_f16;
    float tau;               // 1 / sqrt(D) (block scores)
    float scale_log2;        // tau * log2(e) (attention)
    int* err;
};
int sparse_fused_gmax(int D);
bool sparse_fused_ok(int D, int nb, int K_eff);
cudaError_t launch_sparse_fused(const FusedSparseParams& p, int max_nq, cudaStream_t st);

// Contiguous byte ranges copied by one launch (host-buffer calls: page-locked host memory read
// over the host link into device staging memory). Every address 16-byte aligned.
constexpr int MAX_COPY_SEGS = 3 * 64;
struct CopySegs {
    const void* src[MAX_COPY_SEGS];
    void* dst[MAX_COPY_SEGS];
    int n16[MAX_COPY_SEGS];   // 16-byte units
    int n;
};
cudaError_t launch_copy_segments(const CopySegs& p, cudaStream_t st);

// batched-Q tensor-core prefill (tcgen05)
struct PrefillParams {
    const __half* Q;          // [H_q, M, D] (q_dup: [H_q, M, D/2])
    const uint8_t* kv;        // resident fp16 slot
    float* O;                 // [H_q, M, D] (q_dup: [H_q, M, D/2])
    float* LSE;               // [H_q, M] or nullptr
    int H_q, H_kv, M, N, ntiles, S_suf, causal;
    // q_dup: the slot holds [hi | lo] fp16 pairs of D/2-wide values (the suffix too); each Q row
    // enters the tile twice, [q | q], so S sums both halves, and O is folded: O[c] = O'[c] +
    // O'[c + D/2].
    int q_dup;
    // window > 0: row i sees only positions p_i - window + 1 .. p_i of the prefix and suffix laid
    // end to end, p_i = N + S_suf - M + i (the causal bound, when set, still applies)
    int window;
    float scale_log2;
    int* err;
};
// suf_tiles: the suffix [H_kv, S_suf, D] re-laid out like a resident fp16 slot of suf_ntiles tiles
// partials: split-K workspace (partial_bytes); the launch splits each row tile's keys over CTAs
// when that fills the GPU better, and merges the partials with a second (PDL-chained) kernel.
cudaError_t launch_prefill(const PrefillParams& p, const WorkGroup* grp, int n_groups, const void* suf_tiles,
                           int suf_ntiles, float* partials, size_t partial_bytes, int sms, cudaStream_t st, int D);
bool prefill_supported(int D);

}  // namespace pck
