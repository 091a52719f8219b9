// pck_decode_impl.cuh -- M=1 attention over a resident prefix: split-K ("stream-K") decode with
// the dense suffix and the online-softmax merge fused into the same launch. The templates; they are
// instantiated for D in {64, 128, 256} in pck_decode.cu and for D in {32, 96, 160, 192} in
// pck_decode_xd.cu, so that the two compile in parallel.
//
// Follows "ATTEND.* and ATTEND.PREFIX.*", section "Wire forms": QUERY (M=1), QUERY_FUSED
// (prefix + dense suffix + merge in one dispatch), QUERY_SPARSE_AUTO(_FUSED) (attention
// restricted to selected blocks), with GQA through head_map; and "Shared KV Cache Serving --
// Pion as LLM Memory", section "Wire-protocol details" (LSE of each row for the merge).
//
// Work decomposition. A work item is (query descriptor, kv head, <= 8 q heads of that kv head).
// Every item is a sequence of 16-token resident tiles (the prefix, or the tiles of the selected
// blocks). All items' tiles are concatenated and cut into equal contiguous ranges, one per warp
// ("worker"), so the whole GPU streams the same number of bytes per warp whatever the shapes;
// for sparse items the selector writes the items' tile counts and the workers split them on the
// device. A worker keeps a private ring of shared-memory stages filled by 1-D TMA bulk copies
// (cp.async.bulk, mbarrier completion) and computes each tile with the warp MMA m16n8k16 (fp16
// operands, fp32 accumulation); q and P are split into fp16 hi + lo halves so that the products
// keep fp32 accuracy. Both tiers compute S^T = K q^T with the 16 tokens of the tile as MMA rows
// and the q heads as columns (head h, hi / lo in columns 2h, 2h+1), so that every lane owns
// (2 tokens, 1 head) in the softmax, and O^T += V^T P^T with d as the MMA rows; P moves from the
// score layout into the B operand with one movmatrix.trans per 8 tokens.
//   fp16 slots: the K and V^T A-fragments come straight from the resident core-matrix layout
//     with one ldmatrix.x4 per 16 d (K) or per 16 rows of d (V^T); q stays in registers.
//   mlx4g32 slots: the codes enter the MMA as exact fp16 subnormals (c * 2^-24, one AND per
//     register); the per-group affine terms are applied to the fp32 scores,
//     z = 2^24 s * S + b * sum_d q_d, and for V through P' = p * s and sum_t p_t b_t.
// Each worker writes an (m, l, o) partial per item piece; a second kernel (programmatic
// dependent launch) merges each (item, q head) from its pieces and the dense suffix pieces:
//   m = max m_k, l = sum l_k 2^(m_k - m), O = sum o_k 2^(m_k - m) / l, LSE = (m + log2 l) ln 2.
// Softmax runs in base 2 on log2(e)-prescaled scores; the running max is only moved when a
// tile's max exceeds it by more than 8 (so stored weights stay <= 256), which keeps the
// rescale of the accumulators off the common path and does not change the result.
#pragma once

#include <math.h>

#include <algorithm>
#include <type_traits>

#include "pck_common.cuh"
#include "pck_kernels.h"

namespace pck {

template <int FMT, int D>
struct DCfg {
    static constexpr int KS = D / 16;       // 16-wide k-steps over d
    static constexpr int NG = D / 32;       // mlx4g32 groups per head
    static constexpr int NBV = D / 8;       // PV n-blocks over d
    static constexpr int TB = tile_bytes(FMT, D);
    static constexpr int TPS = FMT == FMT_FP16 ? (D == 32 ? 4 : (D == 64 ? 2 : 1)) : (D == 64 ? 4 : (D == 128 ? 4 : 1));
    static constexpr int STAGE = TPS * TB;
    // D = 512 (fp16): a 32 KB tile per stage, so one stage per warp; four warps' single stages
    // still keep ~100 KB per SM in flight
    static constexpr int NSTAGE = FMT == FMT_FP16 ? (D >= 512 ? 1 : 3) : 2;
    static constexpr int RING = NSTAGE * STAGE;
    // D = 512 (fp16): q's B fragments live in shared memory (KS x 32 lanes x 8 bytes per warp), so
    // that the 128 O accumulators of a lane fit in its registers
    static constexpr bool QS = FMT == FMT_FP16 && D >= 512;
    static constexpr int QBYTES = QS ? (D / 16) * 256 : 0;
    static constexpr int SMEM = DECODE_WARPS * RING + DECODE_WARPS * NSTAGE * 8 + DECODE_WARPS * QBYTES;
};

constexpr float RESCALE_THRESHOLD = 8.0f;   // log2 units
constexpr float LN2 = 0.69314718055994530942f;
// q enters the MMAs as an fp16 hi + lo pair of q * tau * log2(e): the hi part is finite only for
// magnitudes below the largest fp16, so a larger (or non-finite) element of Q is reported through
// the device error word (code 7) instead of silently turning the scores into infinities.
constexpr float Q_LIMIT = 65504.0f;

// ---------------------------------------------------------------- fp16 path (S^T orientation)

// Lane l: tokens t = l/4 and t + 8 of each tile, head q = l%4 of each column block cb (heads
// cb*4 .. cb*4+3 of the item); B fragments of q: column n = l/4 = (head n/2, hi or lo part n%2).
template <int D, int NCB>
struct F16State {
    static constexpr int KS = D / 16;
    static constexpr bool QS = D >= 512;   // q fragments in shared memory (one column block)
    static_assert(!QS || NCB == 1, "D = 512 takes at most 4 q heads per work group");
    uint32_t qb[NCB][QS ? 1 : KS][2];   // B fragments of the item's q (tau*log2e prescaled), hi or lo part
    uint32_t qsm;              // QS: shared-memory address of the warp's q fragments [KS][32 lanes][2]
    float oacc[NCB][KS][4];    // O^T m-tile mt: d = 16mt + l/4 in [0..1], d + 8 in [2..3]; columns
                               // 2q, 2q+1 = (hi, lo) of head cb*4 + q
    float m_ref[NCB];
    float l_part[NCB];
};

// The item's q fragments: every load first (one round trip), then the hi / lo splits.
// (PP: any launch parameter block with q_f16, scale_log2 and err; DS: anything with Q)
template <int D, int NCB, typename PP, typename DS>
__device__ __forceinline__ void start_item_f16(F16State<D, NCB>& st, const PP& p, const DS& ds,
                                               const WorkGroup& wg, int lane) {
    constexpr int KS = D / 16;
    const int q = lane & 3, n = lane >> 2, hl = n >> 1, part = n & 1;
    float2 xq[NCB][KS][2];
#pragma unroll
    for (int cb = 0; cb < NCB; ++cb) {
        const int h = cb * 4 + hl;
        const int qh = h < wg.nq ? wg.qh[h] : -1;
#pragma unroll
        for (int s = 0; s < KS; ++s)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int d0 = 16 * s + 8 * r + 2 * q;
                if (qh < 0) xq[cb][s][r] = make_float2(0.f, 0.f);
                else if (p.q_f16) xq[cb][s][r] = __half22float2(__ldg(reinterpret_cast<const __half2*>(reinterpret_cast<const __half*>(ds.Q) + qh * D + d0)));
                else xq[cb][s][r] = __ldg(reinterpret_cast<const float2*>(reinterpret_cast<const float*>(ds.Q) + qh * D + d0));
            }
    }
    bool bad = false;   // a q element whose prescaled value has no finite fp16 hi part
#pragma unroll
    for (int cb = 0; cb < NCB; ++cb) {
#pragma unroll
        for (int s = 0; s < KS; ++s)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const float x0 = xq[cb][s][r].x * p.scale_log2, x1 = xq[cb][s][r].y * p.scale_log2;
                bad |= !(fabsf(x0) < Q_LIMIT) || !(fabsf(x1) < Q_LIMIT);
                uint32_t hi, lo;
                split_hi_lo(x0, x1, hi, lo);
                if constexpr (F16State<D, NCB>::QS) xq[cb][s][r].x = __uint_as_float(part ? lo : hi);
                else st.qb[cb][s][r] = part ? lo : hi;
            }
        if constexpr (F16State<D, NCB>::QS) {   // each lane reads back only its own entries
#pragma unroll
            for (int s = 0; s < KS; ++s)
                asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(st.qsm + (s * 32 + lane) * 8),
                             "r"(__float_as_uint(xq[cb][s][0].x)), "r"(__float_as_uint(xq[cb][s][1].x))
                             : "memory");
        }
        st.m_ref[cb] = -INFINITY;
        st.l_part[cb] = 0.f;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) st.oacc[cb][mt][0] = st.oacc[cb][mt][1] = st.oacc[cb][mt][2] = st.oacc[cb][mt][3] = 0.f;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) set_err(p.err, 7);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

// One 16-token tile of an fp16 slot in shared memory (resident layout). K part: 2 token groups
// x D/8 d chunks of 128-B core matrices, [8 tokens][8 d] each; V part: D/8 d groups x 2 token
// chunks, [8 d][8 tokens] each. One ldmatrix.x4 gives the A fragment of a k-step of K (tokens x
// 16 d) or of an m-tile of V^T (16 d x tokens).
template <int D>
struct SmemF16Tile {
    uint32_t kp, vp;   // shared-memory addresses of the K and V parts
    int lane;
    __device__ __forceinline__ void ka(int s, uint32_t (&a)[4]) const {
        const int j = lane >> 3;   // core matrix j: token group j & 1, d chunk 2s + (j >> 1)
        ldsm_x4(kp + ((j & 1) * (D / 8) + 2 * s + (j >> 1)) * 128 + (lane & 7) * 16, a);
    }
    __device__ __forceinline__ void va(int mt, uint32_t (&a)[4]) const {
        const int j = lane >> 3;   // core matrix j: d group 2mt + (j & 1), token chunk j >> 1
        ldsm_x4(vp + ((2 * mt + (j & 1)) * 2 + (j >> 1)) * 128 + (lane & 7) * 16, a);
    }
};

// 16 rows of a dense suffix K_suf/V_suf [S_suf, D] copied as they are (row-major, 2 D bytes a
// row) into shared memory: K fragments (tokens x d) by ldmatrix, V^T fragments (d x tokens) by
// ldmatrix.trans of the same row-major 8 x 8 blocks.
template <int D>
struct SmemRowTile {
    uint32_t kp, vp;   // shared-memory addresses of the K rows and the V rows
    int lane;
    __device__ __forceinline__ void ka(int s, uint32_t (&a)[4]) const {
        const int j = lane >> 3;   // matrix j: tokens 8 (j & 1) .., d 16 s + 8 (j >> 1) ..
        ldsm_x4(kp + ((j & 1) * 8 + (lane & 7)) * (2 * D) + (16 * s + 8 * (j >> 1)) * 2, a);
    }
    __device__ __forceinline__ void va(int mt, uint32_t (&a)[4]) const {
        const int j = lane >> 3;   // matrix j: d 16 mt + 8 (j & 1) .., tokens 8 (j >> 1) ..
        const uint32_t addr = vp + ((j >> 1) * 8 + (lane & 7)) * (2 * D) + (16 * mt + 8 * (j & 1)) * 2;
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                     : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]) : "r"(addr));
    }
};

// Dense suffix K_suf/V_suf [S_suf, D] of one kv head, natural layout, read straight from global.
template <int D>
struct GlobalF16Tile {
    const __half* Kg;   // kv head base [S_suf, D]
    const __half* Vg;
    int t0, S, lane;
    __device__ __forceinline__ uint32_t kw(int t, int d) const {
        return t < S ? __ldg(reinterpret_cast<const uint32_t*>(Kg + (size_t)t * D + d)) : 0u;
    }
    __device__ __forceinline__ uint32_t vw(int t, int d) const {
        const unsigned short a = t < S ? __ldg(reinterpret_cast<const unsigned short*>(Vg + (size_t)t * D + d)) : 0;
        const unsigned short b = t + 1 < S ? __ldg(reinterpret_cast<const unsigned short*>(Vg + (size_t)(t + 1) * D + d)) : 0;
        return static_cast<uint32_t>(a) | (static_cast<uint32_t>(b) << 16);
    }
    __device__ __forceinline__ void ka(int s, uint32_t (&a)[4]) const {   // rows: tokens, k: d
        const int g = lane >> 2, d = 16 * s + 2 * (lane & 3), t = t0 + g;
        a[0] = kw(t, d); a[1] = kw(t + 8, d); a[2] = kw(t, d + 8); a[3] = kw(t + 8, d + 8);
    }
    __device__ __forceinline__ void va(int mt, uint32_t (&a)[4]) const {  // rows: d, k: tokens
        const int dd = 16 * mt + (lane >> 2), t = t0 + 2 * (lane & 3);
        a[0] = vw(t, dd); a[1] = vw(t, dd + 8); a[2] = vw(t + 8, dd); a[3] = vw(t + 8, dd + 8);
    }
};

// One 16-token tile: S^T = K q^T (fp32 scores of 2 tokens x 1 head per lane), one online-softmax
// step, then O^T += V^T P^T with P (hi / lo fp16 parts) moved into B fragments by movmatrix.
template <int D, int NCB, typename Src>
__device__ __forceinline__ void tile_f16(F16State<D, NCB>& st, const Src& src, int lane, int valid,
                                         uint32_t head_mask, int nq, int lo = 0) {
    constexpr int KS = D / 16;
    // one column block over 8 or more k-steps: even and odd k-steps accumulate separately, which
    // halves the chain of dependent MMAs a tile waits on
    constexpr int NA = (KS >= 8 && NCB == 1) ? 2 : 1;
    const int q = lane & 3, t0 = lane >> 2;
    float acc[NCB * NA][4];
#pragma unroll
    for (int cb = 0; cb < NCB * NA; ++cb) acc[cb][0] = acc[cb][1] = acc[cb][2] = acc[cb][3] = 0.f;
#pragma unroll
    for (int s = 0; s < KS; ++s) {
        uint32_t a[4];
        src.ka(s, a);
        if constexpr (F16State<D, NCB>::QS) {
            uint32_t b0, b1;
            asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(b0), "=r"(b1) : "r"(st.qsm + (s * 32 + lane) * 8) : "memory");
            mma16816(acc[s % NA], a, b0, b1);
        } else if constexpr (NA == 2) {
            mma16816(acc[s & 1], a, st.qb[0][s][0], st.qb[0][s][1]);
        } else {
#pragma unroll
            for (int cb = 0; cb < NCB; ++cb) mma16816(acc[cb], a, st.qb[cb][s][0], st.qb[cb][s][1]);
        }
    }
    if constexpr (NA == 2) {
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[0][i] += acc[1][i];
    }
    float z[NCB][2];
#pragma unroll
    for (int cb = 0; cb < NCB; ++cb) {
        z[cb][0] = acc[cb][0] + acc[cb][1];   // hi + lo columns
        z[cb][1] = acc[cb][2] + acc[cb][3];
    }
    // masks (warp-uniform test): tokens past the end or before a window, heads the tile does not serve
    const uint32_t heads = nq >= 32 ? 0xFFFFFFFFu : ((1u << nq) - 1u);
    if (valid < 16 || lo > 0 || (head_mask & heads) != heads || nq < 4 * NCB) {
#pragma unroll
        for (int cb = 0; cb < NCB; ++cb) {
            const int h = cb * 4 + q;
            const bool hok = h < nq && ((head_mask >> h) & 1u);
            if (!(hok && t0 < valid && t0 >= lo)) z[cb][0] = -INFINITY;
            if (!(hok && t0 + 8 < valid && t0 + 8 >= lo)) z[cb][1] = -INFINITY;
        }
    }
    // Rescale test on each lane's own maximum: the head's maximum over its 8 lanes passes the
    // threshold exactly when one of the lanes' maxima does, so the cross-lane maximum is only
    // formed when some head rescales.
    bool need_any = false;
    float mt[NCB];
#pragma unroll
    for (int cb = 0; cb < NCB; ++cb) {
        mt[cb] = fmaxf(z[cb][0], z[cb][1]);
        need_any |= mt[cb] > st.m_ref[cb] + RESCALE_THRESHOLD;   // false when the maximum is -inf
    }
    if (__any_sync(0xffffffffu, need_any)) {
#pragma unroll
        for (int cb = 0; cb < NCB; ++cb) {
            float m = mt[cb];                   // lanes with the same q share a head
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
            mt[cb] = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
            const bool need = mt[cb] > st.m_ref[cb] + RESCALE_THRESHOLD;
            const float mnew = need ? mt[cb] : st.m_ref[cb];
            const float alpha = need ? exp2f(st.m_ref[cb] - mnew) : 1.0f;   // exp2(-inf) = 0 on the first tile
            st.l_part[cb] *= alpha;
            st.m_ref[cb] = mnew;
#pragma unroll
            for (int m2 = 0; m2 < KS; ++m2) {   // O^T columns of this lane are head q's
                st.oacc[cb][m2][0] *= alpha; st.oacc[cb][m2][1] *= alpha;
                st.oacc[cb][m2][2] *= alpha; st.oacc[cb][m2][3] *= alpha;
            }
        }
    }
    uint32_t b[NCB][2];
#pragma unroll
    for (int cb = 0; cb < NCB; ++cb) {
        // ex2(-inf) = +0; a head whose m_ref is still -inf has only -inf scores
        const float ms = st.m_ref[cb] == -INFINITY ? 0.f : st.m_ref[cb];
        const float p0 = ex2_approx(z[cb][0] - ms);
        const float p1 = ex2_approx(z[cb][1] - ms);
        st.l_part[cb] += p0 + p1;
        uint32_t h0, h1;
        pack_hilo2(p0, p1, h0, h1);
        b[cb][0] = movmatrix_trans(h0);   // tokens 0..7 as the k rows of B
        b[cb][1] = movmatrix_trans(h1);   // tokens 8..15
    }
#pragma unroll
    for (int m2 = 0; m2 < KS; ++m2) {
        uint32_t a[4];
        src.va(m2, a);
#pragma unroll
        for (int cb = 0; cb < NCB; ++cb) mma16816(st.oacc[cb][m2], a, b[cb][0], b[cb][1]);
    }
}

// Partial of the item piece: for every head h of the item, [m, l, o[0..D)].
template <int D, int NCB>
__device__ __forceinline__ void write_partial_f16(F16State<D, NCB>& st, float* P, int nq, int lane) {
    constexpr int KS = D / 16;
    const int q = lane & 3, l4 = lane >> 2;
#pragma unroll
    for (int cb = 0; cb < NCB; ++cb) {
        const int hq = cb * 4 + q;
        float l = st.l_part[cb];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        if (hq < nq) {
            float* ph = P + hq * partial_stride(D);
            if (lane < 4) {
                ph[0] = st.m_ref[cb];
                ph[1] = l;
            }
#pragma unroll
            for (int m2 = 0; m2 < KS; ++m2) {   // columns 2q (hi) and 2q+1 (lo) hold the same head
                ph[PARTIAL_O + 16 * m2 + l4] = st.oacc[cb][m2][0] + st.oacc[cb][m2][1];
                ph[PARTIAL_O + 16 * m2 + l4 + 8] = st.oacc[cb][m2][2] + st.oacc[cb][m2][3];
            }
        }
    }
}

// ---------------------------------------------------------------- mlx4g32 path (S^T orientation)

// Lane l: tokens t = l/4 and t + 8 of each tile, head q = l%4 of each column block cb (heads
// cb*4 .. cb*4+3 of the item); B fragments of q: column n = l/4 = (head hl = n/2, part = n%2).
template <int D, int NCB>
struct I4State {
    static constexpr int KS = D / 16, NG = D / 32, NBV = D / 8;
    uint32_t qb[NCB][KS][2];   // B fragments of the item's q (tau*log2e prescaled), hi or lo part
    float qs[NCB][NG];         // sum over the group's d of the lane's head q (prescaled)
    float oacc[NCB][KS][4];    // O^T m-tile mt: d = 16mt + l/4 in [0..1], d + 8 in [2..3]; columns
                               // 2q, 2q+1 = (hi, lo) of head cb*4 + q
    float bacc[NCB][NG];       // sum_t p_t * bias_t of the lane's head, per group
    float m_ref[NCB];
    float l_part[NCB];
};

template <int D, int NCB>
__device__ __forceinline__ void start_item_i4(I4State<D, NCB>& st, const DecodeParams& p, const DecodeDesc& ds,
                                              const WorkGroup& wg, int lane) {
    using S = I4State<D, NCB>;
    const int q = lane & 3, n = lane >> 2, hl = n >> 1, part = n & 1;
    bool bad = false;   // a q element whose prescaled value has no finite fp16 hi part
#pragma unroll
    for (int cb = 0; cb < NCB; ++cb) {
        const int h = cb * 4 + hl;
        const int qh = h < wg.nq ? wg.qh[h] : -1;
        float gsum[S::NG];
#pragma unroll
        for (int g = 0; g < S::NG; ++g) gsum[g] = 0.f;
        float2 xq[S::KS][2];   // every load first (one round trip)
#pragma unroll
        for (int s = 0; s < S::KS; ++s)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int d0 = 16 * s + 8 * r + 2 * q;
                if (qh < 0) xq[s][r] = make_float2(0.f, 0.f);
                else if (p.q_f16) xq[s][r] = __half22float2(__ldg(reinterpret_cast<const __half2*>(reinterpret_cast<const __half*>(ds.Q) + qh * D + d0)));
                else xq[s][r] = __ldg(reinterpret_cast<const float2*>(reinterpret_cast<const float*>(ds.Q) + qh * D + d0));
            }
#pragma unroll
        for (int s = 0; s < S::KS; ++s) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const float x0 = xq[s][r].x * p.scale_log2, x1 = xq[s][r].y * p.scale_log2;
                bad |= !(fabsf(x0) < Q_LIMIT) || !(fabsf(x1) < Q_LIMIT);
                gsum[s >> 1] += x0 + x1;
                uint32_t hi, lo;
                split_hi_lo(x0, x1, hi, lo);
                st.qb[cb][s][r] = part ? lo : hi;
            }
        }
        // gsum: this lane's 8 of the group's 32 d of head hl; the 4 lanes q = 0..3 of a column
        // hold all 32, and lane 8*h' (column 2h') holds head h' -> the lane's S^T head q.
#pragma unroll
        for (int g = 0; g < S::NG; ++g) {
            float v = gsum[g];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            st.qs[cb][g] = __shfl_sync(0xffffffffu, v, 8 * q);
            st.bacc[cb][g] = 0.f;
        }
        st.m_ref[cb] = -INFINITY;
        st.l_part[cb] = 0.f;
#pragma unroll
        for (int mt = 0; mt < S::KS; ++mt) st.oacc[cb][mt][0] = st.oacc[cb][mt][1] = st.oacc[cb][mt][2] = st.oacc[cb][mt][3] = 0.f;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) set_err(p.err, 7);
}

// NT (1, 2 or 4) consecutive 16-token tiles of a kv head: scores of all NT*16 tokens, one online
// softmax step, then O += P' V for each tile.
template <int D, int NCB, int NT>
__device__ __forceinline__ void tile_i4(I4State<D, NCB>& st, const uint8_t* tile0, int lane, int valid0,
                                        uint32_t head_mask, int nq, int lo0 = 0) {
    using S = I4State<D, NCB>;
    constexpr int NG = S::NG, KS = S::KS, TB = 20 * D;
    const int q = lane & 3, t0 = lane >> 2;
    uint32_t kw[NT][KS], vw[NT][KS];
    uint32_t ks0[NT][NG], ks1[NT][NG], vs0[NT][NG], vs1[NT][NG];   // (scale, bias) of tokens t0, t0+8
#pragma unroll
    for (int x = 0; x < NT; ++x) {
        const uint8_t* tile = tile0 + x * TB;
        const uint32_t* ksb = reinterpret_cast<const uint32_t*>(tile + 8 * D);
        const uint32_t* vsb = reinterpret_cast<const uint32_t*>(tile + 18 * D);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {   // 16-byte loads: consecutive lanes, consecutive 16 B
            const uint4 v = *reinterpret_cast<const uint4*>(tile + (c * 32 + lane) * 16);
            kw[x][4 * c] = v.x; kw[x][4 * c + 1] = v.y; kw[x][4 * c + 2] = v.z; kw[x][4 * c + 3] = v.w;
            const uint4 u = *reinterpret_cast<const uint4*>(tile + 10 * D + (c * 32 + lane) * 16);
            vw[x][4 * c] = u.x; vw[x][4 * c + 1] = u.y; vw[x][4 * c + 2] = u.z; vw[x][4 * c + 3] = u.w;
        }
#pragma unroll
        for (int g = 0; g < NG; g += 2) {
            const uint2 a = *reinterpret_cast<const uint2*>(ksb + t0 * NG + g);
            const uint2 b = *reinterpret_cast<const uint2*>(ksb + (t0 + 8) * NG + g);
            const uint2 c = *reinterpret_cast<const uint2*>(vsb + t0 * NG + g);
            const uint2 d = *reinterpret_cast<const uint2*>(vsb + (t0 + 8) * NG + g);
            ks0[x][g] = a.x; ks0[x][g + 1] = a.y; ks1[x][g] = b.x; ks1[x][g + 1] = b.y;
            vs0[x][g] = c.x; vs0[x][g + 1] = c.y; vs1[x][g] = d.x; vs1[x][g + 1] = d.y;
        }
    }
    // ---- scores: z[x][cb][0] token 16x + t0, z[x][cb][1] token 16x + t0 + 8 (head q of block cb)
    float z[NT][NCB][2];
#pragma unroll
    for (int x = 0; x < NT; ++x) {
        float zs0[NCB], zs1[NCB], zb0[NCB], zb1[NCB];
#pragma unroll
        for (int cb = 0; cb < NCB; ++cb) zs0[cb] = zs1[cb] = zb0[cb] = zb1[cb] = 0.f;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            float acc[NCB][4];
#pragma unroll
            for (int cb = 0; cb < NCB; ++cb) acc[cb][0] = acc[cb][1] = acc[cb][2] = acc[cb][3] = 0.f;
#pragma unroll
            for (int ss = 0; ss < 2; ++ss) {
                const int s = 2 * g + ss;
                uint32_t a[4];
                unpack_word(kw[x][s], a[0], a[1], a[2], a[3]);
#pragma unroll
                for (int cb = 0; cb < NCB; ++cb) mma16816(acc[cb], a, st.qb[cb][s][0], st.qb[cb][s][1]);
            }
            const float2 sb0 = __half22float2(u32_as_h2(ks0[x][g]));
            const float2 sb1 = __half22float2(u32_as_h2(ks1[x][g]));
#pragma unroll
            for (int cb = 0; cb < NCB; ++cb) {
                zs0[cb] = fmaf(sb0.x, acc[cb][0] + acc[cb][1], zs0[cb]);
                zs1[cb] = fmaf(sb1.x, acc[cb][2] + acc[cb][3], zs1[cb]);
                zb0[cb] = fmaf(sb0.y, st.qs[cb][g], zb0[cb]);
                zb1[cb] = fmaf(sb1.y, st.qs[cb][g], zb1[cb]);
            }
        }
#pragma unroll
        for (int cb = 0; cb < NCB; ++cb) {
            z[x][cb][0] = fmaf(zs0[cb], 16777216.0f, zb0[cb]);     // 2^24: codes entered as c * 2^-24
            z[x][cb][1] = fmaf(zs1[cb], 1048576.0f, zb1[cb]);      // 2^20: rows t0+8 hold 16 c * 2^-24
        }
    }
    // masks (warp-uniform test): tokens past the end of the prefix or before a window, heads the
    // chunk does not serve
    const uint32_t heads = nq >= 32 ? 0xFFFFFFFFu : ((1u << nq) - 1u);
    if (valid0 < 16 * NT || lo0 > 0 || (head_mask & heads) != heads || nq < 4 * NCB) {
#pragma unroll
        for (int x = 0; x < NT; ++x) {
            const int va = valid0 - 16 * x, lx = lo0 - 16 * x;
#pragma unroll
            for (int cb = 0; cb < NCB; ++cb) {
                const int h = cb * 4 + q;
                const bool hok = h < nq && ((head_mask >> h) & 1u);
                if (!(hok && t0 < va && t0 >= lx)) z[x][cb][0] = -INFINITY;
                if (!(hok && t0 + 8 < va && t0 + 8 >= lx)) z[x][cb][1] = -INFINITY;
            }
        }
    }
    // ---- online softmax step over the NT*16 tokens (lanes with the same q share a head)
    // (the rescale test runs on each lane's own maximum; the cross-lane maximum only when some
    //  head rescales, as in tile_f16)
    bool need_any = false;
    float mt[NCB];
#pragma unroll
    for (int cb = 0; cb < NCB; ++cb) {
        float m = fmaxf(z[0][cb][0], z[0][cb][1]);
#pragma unroll
        for (int x = 1; x < NT; ++x) m = fmaxf(m, fmaxf(z[x][cb][0], z[x][cb][1]));
        mt[cb] = m;
        need_any |= m > st.m_ref[cb] + RESCALE_THRESHOLD;
    }
    if (__any_sync(0xffffffffu, need_any)) {
#pragma unroll
        for (int cb = 0; cb < NCB; ++cb) {
            float m = mt[cb];
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
            mt[cb] = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
            const bool need = mt[cb] > st.m_ref[cb] + RESCALE_THRESHOLD;
            const float mnew = need ? mt[cb] : st.m_ref[cb];
            const float alpha = need ? exp2f(st.m_ref[cb] - mnew) : 1.0f;   // head q's factor
            st.l_part[cb] *= alpha;
#pragma unroll
            for (int g = 0; g < NG; ++g) st.bacc[cb][g] *= alpha;
            st.m_ref[cb] = mnew;
#pragma unroll
            for (int m2 = 0; m2 < KS; ++m2) {   // O^T columns of this lane are head q's
                st.oacc[cb][m2][0] *= alpha; st.oacc[cb][m2][1] *= alpha;
                st.oacc[cb][m2][2] *= alpha; st.oacc[cb][m2][3] *= alpha;
            }
        }
    }
    float pr[NT][NCB][2];
#pragma unroll
    for (int x = 0; x < NT; ++x)
#pragma unroll
        for (int cb = 0; cb < NCB; ++cb) {
            // ex2(-inf) = +0; a head whose m_ref is still -inf has only -inf scores (any finite
            // one would have moved it), so 0 stands in for it there
            const float ms = st.m_ref[cb] == -INFINITY ? 0.f : st.m_ref[cb];
#pragma unroll
            for (int y = 0; y < 2; ++y) pr[x][cb][y] = ex2_approx(z[x][cb][y] - ms);
            st.l_part[cb] += pr[x][cb][0] + pr[x][cb][1];
        }
    // ---- O^T += V^T P'^T per tile and group of 32 d (P' = p * scale of the token's group):
    //      A = V codes (d as rows), B = P' of the 16 tokens x (head, hi/lo) columns
#pragma unroll
    for (int x = 0; x < NT; ++x) {
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            const float2 sv0 = __half22float2(u32_as_h2(vs0[x][g]));
            const float2 sv1 = __half22float2(u32_as_h2(vs1[x][g]));
            uint32_t b[NCB][2];
#pragma unroll
            for (int cb = 0; cb < NCB; ++cb) {
                st.bacc[cb][g] = fmaf(pr[x][cb][0], sv0.y, fmaf(pr[x][cb][1], sv1.y, st.bacc[cb][g]));
                uint32_t h0, h1;
                pack_hilo2(pr[x][cb][0] * sv0.x, pr[x][cb][1] * sv1.x, h0, h1);
                b[cb][0] = movmatrix_trans(h0);   // tokens 0..7
                b[cb][1] = movmatrix_trans(h1);   // tokens 8..15
            }
#pragma unroll
            for (int ww = 0; ww < 2; ++ww) {
                const int m2 = 2 * g + ww;          // m-tile of 16 d
                uint32_t a[4];
                unpack_word(vw[x][m2], a[0], a[1], a[2], a[3]);
#pragma unroll
                for (int cb = 0; cb < NCB; ++cb) mma16816(st.oacc[cb][m2], a, b[cb][0], b[cb][1]);
            }
        }
    }
}

// Partial of the item piece: for every head h of the item, [m, l, o[0..D)] with o already in
// real units (2^24 and the V biases applied).
template <int D, int NCB>
__device__ __forceinline__ void write_partial_i4(I4State<D, NCB>& st, float* P, int nq, int lane) {
    using S = I4State<D, NCB>;
    const int q = lane & 3, l4 = lane >> 2;
#pragma unroll
    for (int cb = 0; cb < NCB; ++cb) {
        const int hq = cb * 4 + q;   // this lane's head for l, bias and the O^T columns
        float l = st.l_part[cb];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        float bsum[S::NG];
#pragma unroll
        for (int g = 0; g < S::NG; ++g) {
            float v = st.bacc[cb][g];
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            v += __shfl_xor_sync(0xffffffffu, v, 8);
            v += __shfl_xor_sync(0xffffffffu, v, 16);
            bsum[g] = v;
        }
        if (hq < nq) {
            float* ph = P + hq * partial_stride(D);
            if (lane < 4) {
                ph[0] = st.m_ref[cb];
                ph[1] = l;
            }
#pragma unroll
            for (int m2 = 0; m2 < S::KS; ++m2) {
                const float b = bsum[m2 / 2];
                const int d = 16 * m2 + l4;
                // columns 2q (hi) and 2q+1 (lo) hold the same head; rows d+8 carry 16 c
                ph[PARTIAL_O + d] = fmaf(st.oacc[cb][m2][0] + st.oacc[cb][m2][1], 16777216.0f, b);
                ph[PARTIAL_O + d + 8] = fmaf(st.oacc[cb][m2][2] + st.oacc[cb][m2][3], 1048576.0f, b);
            }
        }
    }
}

// ---------------------------------------------------------------- pieces, tickets and the merge

// Units per prefix worker: host-computed when dense; for a sparse launch, the selector's total
// split over all the prefix workers.
__device__ __forceinline__ int worker_units(const DecodeParams& p, int total) {
    return p.sparse ? max(1, (total + p.n_workers - 1) / p.n_workers) : p.tpw;
}

// The item's units [s, e) and the first prefix worker w0 whose range meets them; the pieces of
// the item are those of workers w0 .. w0 + npref - 1 (npref = 0 when the item has no units).
__device__ __forceinline__ void item_range(const DecodeParams& p, int item, int& w0, int& npref) {
    const int d = item / p.n_groups, grp = item - d * p.n_groups;
    int s = 0, e = 0, tpw = 1;
    if (p.sparse) {
        const int n_items = p.n_desc * p.n_groups;
        s = min(max(__ldcg(p.item_base + item), 0), p.max_units);
        e = min(max(__ldcg(p.item_base + item + 1), s), p.max_units);
        tpw = worker_units(p, min(max(__ldcg(p.item_base + n_items), 0), p.max_units));
    } else if (p.aligned) {   // the item's whole pieces
        w0 = p.wbase[d] + grp * p.ppi[d];
        npref = p.ppi[d];
        return;
    } else {
        s = p.desc[d].tile_off + grp * p.desc[d].vtiles;
        e = s + p.desc[d].vtiles;
        tpw = p.tpw;
    }
    w0 = s / tpw;
    npref = e > s ? (e - 1) / tpw - w0 + 1 : 0;
}

// Merge of one (item, q head). Pieces are taken in batches of BP (16 float4 of o per lane, 32
// at D = 256, where few items mean few warps); all of a batch's loads (m and l of the lane's
// piece, and every o) are issued before any is used, so a batch costs one L2 round trip. Batches are combined with an
// online rescale; within a batch the weights 2^(m_k - M) are broadcast by shuffles. Partials are
// read through L2 (__ldcg).
template <int D>
__device__ void merge_item_head(const DecodeParams& p, int item, int h, int lane, int w0, int npref) {
    const int d = item / p.n_groups, grp = item - d * p.n_groups;
    const DecodeDesc& ds = p.desc[d];
    const WorkGroup& wg = p.grp[grp];
    const int n_items = p.n_desc * p.n_groups;
    const int npieces = npref + p.n_suf;
    constexpr int PSTR = GMAX * partial_stride(D);
    auto piece = [&](int k) -> const float* {
        const int slot = k < npref ? (w0 + k + item) : (p.n_workers + n_items + item * p.n_suf + (k - npref));
        return p.partials + (size_t)slot * PSTR + h * partial_stride(D);
    };
    constexpr int F4 = D / 4;                      // float4 of o per piece
    constexpr int LPP = F4 >= 32 ? 32 : (F4 > 16 ? 32 : (F4 > 8 ? 16 : 8));   // lanes per piece (a power of 2)
    constexpr int PPS = 32 / LPP;                  // pieces per warp-wide load
    constexpr int V4 = (F4 + LPP - 1) / LPP;       // float4 per lane per piece
    constexpr int NB0 = 32 / PPS < 16 ? 32 / PPS : 16;
    constexpr int NB = V4 > 2 ? NB0 * 2 / V4 : NB0;     // warp-wide loads per batch (<= 32 float4 per lane)
    constexpr int BP = NB * PPS;                   // pieces per batch (<= 32: one lane per piece's (m, l))
    const int sub = lane / LPP, dl = lane % LPP;
    float M = -INFINITY, L = 0.f;                  // L: this lane's share (lanes over pieces)
    float4 acc[V4];
#pragma unroll
    for (int v = 0; v < V4; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c = 0; c < npieces; c += BP) {
        const int nk = min(BP, npieces - c);
        float mk = -INFINITY, lk = 0.f;
        if (lane < nk) {
            const float2 ml = __ldcg(reinterpret_cast<const float2*>(piece(c + lane)));
            mk = ml.x;
            lk = ml.y;
        }
        float4 xs[NB][V4];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const int jj = b * PPS + sub;
            if (jj < nk) {
                const float4* ph = reinterpret_cast<const float4*>(piece(c + jj) + PARTIAL_O) + dl;
#pragma unroll
                for (int v = 0; v < V4; ++v)
                    xs[b][v] = dl + v * LPP < F4 ? __ldcg(ph + v * LPP) : make_float4(0.f, 0.f, 0.f, 0.f);
            } else {
#pragma unroll
                for (int v = 0; v < V4; ++v) xs[b][v] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        float Mb = mk;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) Mb = fmaxf(Mb, __shfl_xor_sync(0xffffffffu, Mb, o));
        const float Mn = fmaxf(M, Mb);
        if (Mn != -INFINITY) {
            const float r = M == -INFINITY ? 0.f : exp2f(M - Mn);   // rescale of earlier batches
            L *= r;
#pragma unroll
            for (int v = 0; v < V4; ++v) { acc[v].x *= r; acc[v].y *= r; acc[v].z *= r; acc[v].w *= r; }
            M = Mn;
        }
        const float wk = mk == -INFINITY ? 0.f : exp2f(mk - M);
        L = fmaf(wk, lk, L);
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const float w = __shfl_sync(0xffffffffu, wk, (b * PPS + sub) & 31);
#pragma unroll
            for (int v = 0; v < V4; ++v) {
                acc[v].x = fmaf(w, xs[b][v].x, acc[v].x);
                acc[v].y = fmaf(w, xs[b][v].y, acc[v].y);
                acc[v].z = fmaf(w, xs[b][v].z, acc[v].z);
                acc[v].w = fmaf(w, xs[b][v].w, acc[v].w);
            }
        }
    }
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) L += __shfl_xor_sync(0xffffffffu, L, x);
#pragma unroll
    for (int x = LPP; x < 32; x <<= 1) {   // sum the pieces' partial sums across lane groups
#pragma unroll
        for (int v = 0; v < V4; ++v) {
            acc[v].x += __shfl_xor_sync(0xffffffffu, acc[v].x, x);
            acc[v].y += __shfl_xor_sync(0xffffffffu, acc[v].y, x);
            acc[v].z += __shfl_xor_sync(0xffffffffu, acc[v].z, x);
            acc[v].w += __shfl_xor_sync(0xffffffffu, acc[v].w, x);
        }
    }
    const int qh = wg.qh[h];
    const float inv = L > 0.f ? 1.0f / L : 0.f;
    if (sub == 0) {
#pragma unroll
        for (int v = 0; v < V4; ++v)
            if (dl + v * LPP < F4)
                reinterpret_cast<float4*>(ds.O + (size_t)qh * D)[dl + v * LPP] =
                    make_float4(acc[v].x * inv, acc[v].y * inv, acc[v].z * inv, acc[v].w * inv);
    }
    if (lane == 0 && ds.LSE) ds.LSE[qh] = L > 0.f ? (M + log2f(L)) * LN2 : -INFINITY;
}

// Second kernel of a decode: one warp per (item, q head) slot, GMAX slots per item (the grid
// covers them all). Launched with programmatic dependent launch; it waits for the decode grid
// (partials complete and visible) before reading them. A dense launch's piece range depends on
// launch parameters only and is found before that wait; a sparse one's comes from the unit
// offsets the selection grid wrote, so after it.
template <int D>
__global__ void __launch_bounds__(256) merge_kernel(const __grid_constant__ DecodeParams p) {
    const int lane = threadIdx.x & 31;
    const int wi = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int item = wi / GMAX, h = wi - item * GMAX;
    // the next kernel of the stream may be scheduled now: a decode then sets up its workers from
    // its launch parameters and fills its first ring stages with resident tiles while this merge
    // runs, and waits for it before reading anything else
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const bool live = wi < p.n_desc * p.n_groups * GMAX && h < p.grp[item % p.n_groups].nq;   // warp-uniform
    int w0 = 0, npref = 0;
    if (live && !p.sparse) item_range(p, item, w0, npref);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (!live) return;
    if (p.sparse) item_range(p, item, w0, npref);
    merge_item_head<D>(p, item, h, lane, w0, npref);
}

template <int D, int NCB>
__device__ void finish_piece_f16(F16State<D, NCB>& st, const DecodeParams& p, int item, int slot, int lane) {
    write_partial_f16<D, NCB>(st, p.partials + (size_t)slot * GMAX * partial_stride(D), p.grp[item % p.n_groups].nq, lane);
}

template <int D, int NCB>
__device__ void finish_piece_i4(I4State<D, NCB>& st, const DecodeParams& p, int item, int slot, int lane) {
    const int grp = item % p.n_groups;
    write_partial_i4<D, NCB>(st, p.partials + (size_t)slot * GMAX * partial_stride(D), p.grp[grp].nq, lane);
}

// ---------------------------------------------------------------- tile cursor over a worker range

// A worker walks a contiguous range of units. Dense: a unit is one of the item's resident tiles
// (items laid end to end, host-computed ranges). Sparse: a unit is one tile of a block that the
// item's selection list holds, in list order; the selector wrote each item's first unit
// (item_base), and the workers split [0, total) evenly on the device. The cursor keeps what a
// chunk needs of the current item in registers, so a chunk reads no launch parameter.
struct Cursor {
    int t, t_end;            // current unit, end of the worker's range
    int item, d, grp;        // current item (= d * n_groups + grp)
    int item_start, item_end;
    int ntiles, N, nq;
    int tile0, t_lo;         // the item's first resident tile and first visible token (a window)
    const uint8_t* kbase;    // fp16: K region of the item's kv head; mlx4g32: the kv head's tiles
    size_t vofs;             // fp16: bytes from the K region to the V region
    int sel_blk, sel_msk;    // sparse, lists of <= 32 blocks: lane l holds entry l of the item's list
    int win, win_lo;         // sparse: lane l holds item_base[win_lo + l]
};

struct Chunk {
    int item, d, grp;
    int tile;     // first real tile (within the kv head) of the chunk
    int nreal;    // tiles to copy and compute
    int valid;    // tokens of the prefix from the chunk's first token on
    int lo;       // tokens of the chunk's first tile below the window (<= 0: none)
    int nq;       // q heads of the item
    uint32_t mask;// bit h: local q head h attends to this chunk's tokens
    bool last;    // last chunk of this worker's piece of the item
    const uint8_t* src;   // mlx4g32: the tiles; fp16: the K region part
    const uint8_t* src2;  // fp16: the V region part
};

__device__ __forceinline__ int units_total(const DecodeParams& p) {
    const int n_items = p.n_desc * p.n_groups;
    return min(max(__ldcg(p.item_base + n_items), 0), p.max_units);
}

// item_base[i], clamped into [0, max_units] (read from the lane window, reloaded when i leaves it)
__device__ __forceinline__ int cursor_base(const DecodeParams& p, Cursor& c, int i) {
    const int n_items = p.n_desc * p.n_groups;
    if (i - c.win_lo > 31 || i < c.win_lo) {
        const int lane = threadIdx.x & 31;
        c.win_lo = i;
        c.win = min(max(__ldcg(p.item_base + min(i + lane, n_items)), 0), p.max_units);
    }
    return __shfl_sync(0xffffffffu, c.win, i - c.win_lo);
}

template <int FMT, int D>
__device__ __forceinline__ void cursor_set_item(const DecodeParams& p, Cursor& c) {
    const DecodeDesc& ds = p.desc[c.d];
    const WorkGroup& wg = p.grp[c.grp];
    c.ntiles = ds.ntiles;
    c.N = ds.N;
    c.nq = wg.nq;
    c.tile0 = ds.tile0;
    c.t_lo = ds.t_lo;
    if constexpr (FMT == FMT_FP16) {
        c.vofs = fp16_region_bytes(ds.ntiles, D);
        c.kbase = ds.kv + (size_t)wg.g * 2 * c.vofs;
    } else {
        c.vofs = 0;
        c.kbase = ds.kv + (size_t)wg.g * ds.ntiles * tile_bytes(FMT_I4, D);
    }
    if (FMT == FMT_FP16 && p.sparse && p.sel_max <= 32) {
        const int lane = threadIdx.x & 31;
        const int base = c.grp * p.sel_max;
        c.sel_blk = lane < p.sel_max ? ds.sel_blocks[base + lane] : -1;
        c.sel_msk = lane < p.sel_max ? ds.sel_mask[base + lane] : 0;
    }
}

// Sparse: make `i` (or the first non-empty item after it) the current item; units >= t exist.
template <int FMT, int D>
__device__ __forceinline__ void cursor_enter_sparse(const DecodeParams& p, Cursor& c, int i) {
    const int n_items = p.n_desc * p.n_groups;
    int e = cursor_base(p, c, i + 1);
    while (e <= c.t && i + 1 < n_items) {   // skip items that end at or before t (empty ones)
        ++i;
        e = cursor_base(p, c, i + 1);
    }
    c.item = i;
    c.item_start = cursor_base(p, c, i);
    c.item_end = e;
    c.d = i / p.n_groups;
    c.grp = i - c.d * p.n_groups;
    cursor_set_item<FMT, D>(p, c);
}

// Position a cursor at unit t (the first of worker w's range).
template <int FMT, int D>
__device__ __forceinline__ void cursor_seek(const DecodeParams& p, Cursor& c) {
    if (FMT != FMT_FP16 || !p.sparse) {
        int d = 0;
        while (d + 1 < p.n_desc && p.desc[d + 1].tile_off <= c.t) ++d;
        const int vt = p.desc[d].vtiles;
        const int grp = (c.t - p.desc[d].tile_off) / vt;
        c.d = d;
        c.grp = grp;
        c.item = d * p.n_groups + grp;
        c.item_start = p.desc[d].tile_off + grp * vt;
        c.item_end = c.item_start + vt;
        cursor_set_item<FMT, D>(p, c);
        return;
    }
    // the largest item i with item_base[i] <= t: a 32-way search over item_base; its last step
    // loads item_base[lo .. lo + 31], which then serves as the cursor's window
    const int n_items = p.n_desc * p.n_groups;
    const int lane = threadIdx.x & 31;
    int lo = 0, hi = n_items;
    while (hi - lo > 31) {
        const int step = (hi - lo + 31) / 32;
        const int idx = lo + lane * step;
        const bool ok = idx < hi && min(max(__ldcg(p.item_base + idx), 0), p.max_units) <= c.t;
        const unsigned b = __ballot_sync(0xffffffffu, ok);   // a prefix of the lanes (lane 0 always)
        const int k = 31 - __clz(b | 1u);
        lo += k * step;
        hi = min(hi, lo + step);
    }
    c.win_lo = lo;
    c.win = min(max(__ldcg(p.item_base + min(lo + lane, n_items)), 0), p.max_units);
    const unsigned b = __ballot_sync(0xffffffffu, lo + lane < hi && c.win <= c.t);
    cursor_enter_sparse<FMT, D>(p, c, lo + 31 - __clz(b | 1u));
}

template <int FMT, int D, int TPS, int TB>
__device__ __forceinline__ bool cursor_next(const DecodeParams& p, Cursor& c, Chunk& ch) {
    if (c.t >= c.t_end) return false;
    constexpr bool CAN_SPARSE = FMT == FMT_FP16;   // sparse launches hold fp16 slots
    if (c.t >= c.item_end) {
        if (!CAN_SPARSE || !p.sparse) {
            if (++c.grp == p.n_groups) { c.grp = 0; ++c.d; }
            c.item = c.d * p.n_groups + c.grp;
            c.item_start = p.desc[c.d].tile_off + c.grp * p.desc[c.d].vtiles;
            c.item_end = c.item_start + p.desc[c.d].vtiles;
            cursor_set_item<FMT, D>(p, c);
        } else {
            cursor_enter_sparse<FMT, D>(p, c, c.item + 1);
        }
    }
    const int local = c.t - c.item_start;
    const int lim = min(c.t_end, c.item_end) - c.t;
    int n;
    if (!CAN_SPARSE || !p.sparse) {
        n = min(TPS, lim);
        ch.tile = c.tile0 + local;
        ch.nreal = n;
        ch.mask = 0xFFu;
    } else {
        // unit `local` of the item: tile `local % tpb` of the block in list slot `local / tpb`
        // (every slot before the item's last holds a whole block; the last may be the ragged end)
        const int slot = min(max(local / p.tiles_per_block, 0), p.sel_max - 1);
        const int within = local - (local / p.tiles_per_block) * p.tiles_per_block;
        n = 1;
        int blk, msk;
        if (p.sel_max <= 32) {
            blk = __shfl_sync(0xffffffffu, c.sel_blk, slot & 31);
            msk = __shfl_sync(0xffffffffu, c.sel_msk, slot & 31);
        } else {
            const DecodeDesc& ds = p.desc[c.d];
            blk = ds.sel_blocks[c.grp * p.sel_max + slot];
            msk = ds.sel_mask[c.grp * p.sel_max + slot];
        }
        ch.tile = max(blk, 0) * p.tiles_per_block + within;
        ch.nreal = blk >= 0 && within >= 0 && ch.tile < c.ntiles ? 1 : 0;
        ch.mask = static_cast<uint32_t>(msk);
    }
    ch.item = c.item;
    ch.d = c.d;
    ch.grp = c.grp;
    ch.nq = c.nq;
    ch.valid = c.N - ch.tile * TILE_TOK;
    ch.lo = c.t_lo - ch.tile * TILE_TOK;
    if constexpr (FMT == FMT_FP16) {
        ch.src = c.kbase + (size_t)ch.tile * 32 * D;
        ch.src2 = c.kbase + c.vofs + (size_t)ch.tile * 32 * D;
    } else {
        ch.src = c.kbase + (size_t)ch.tile * TB;
        ch.src2 = nullptr;
    }
    c.t += n;
    ch.last = (c.t == c.item_end) || (c.t == c.t_end);
    return true;
}

// ---------------------------------------------------------------- workers

// This grid may be launched before the previous kernel of the stream has finished (programmatic
// dependence): wait for it before reading anything it may have written, then let the merge
// kernel be scheduled (it still waits for this whole grid before reading a partial).
__device__ __forceinline__ void grid_dep_wait_then_release() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <int FMT, int D, int NCB>
__device__ void prefix_worker(const DecodeParams& p, int w, int lane, uint8_t* ring, uint64_t* bars, uint8_t* qarea) {
    using C = DCfg<FMT, D>;
    using StateT = std::conditional_t<FMT == FMT_FP16, F16State<D, NCB>, I4State<D, NCB>>;
    Cursor cons;
    const bool sparse = FMT == FMT_FP16 && p.sparse;
    if (sparse) grid_dep_wait_then_release();   // the unit offsets come from the previous grid
    const int total = FMT == FMT_FP16 && p.sparse ? units_total(p) : p.total_tiles;
    if ((FMT == FMT_FP16 && p.sparse) || !p.aligned) {
        const int tpw = worker_units(p, total);
        cons.t = w * tpw;
        cons.t_end = min(total, cons.t + tpw);
    } else {   // dense, aligned: piece k of item (d, grp), found from the descriptors' first workers
        int d = 0;
        while (d + 1 < p.n_desc && p.wbase[d + 1] <= w) ++d;
        const int r = w - p.wbase[d], ppi = p.ppi[d], vt = p.desc[d].vtiles;
        const int grp = r / ppi, k = r - grp * ppi;
        const int ps = (vt + ppi - 1) / ppi;
        const int s0 = p.desc[d].tile_off + grp * vt;
        cons.t = s0 + k * ps;
        cons.t_end = min(s0 + vt, cons.t + ps);
    }
    if (cons.t >= cons.t_end) {
        if (!sparse) grid_dep_wait_then_release();
        return;
    }
    cursor_seek<FMT, D>(p, cons);
    Cursor prod = cons;

    const uint32_t ring_s = smem_u32(ring);
    const uint32_t bar_s = smem_u32(bars);
    if (lane == 0) {
        for (int s = 0; s < C::NSTAGE; ++s) mbar_init(bar_s + 8 * s, 1);
        fence_mbar_init();
    }
    __syncwarp();

    // the slot's tiles are read once per launch: first out of L2
    const uint64_t pol = l2_evict_first();
    auto issue = [&](const Chunk& c, int s) {
        if (lane == 0) {
            if (c.nreal > 0) {
                mbar_arrive_expect_tx(bar_s + 8 * s, c.nreal * C::TB);
                if constexpr (FMT == FMT_FP16) {
                    const uint32_t half = c.nreal * 32 * D;
                    bulk_g2s_hint(ring_s + s * C::STAGE, c.src, half, bar_s + 8 * s, pol);
                    bulk_g2s_hint(ring_s + s * C::STAGE + C::STAGE / 2, c.src2, half, bar_s + 8 * s, pol);
                } else {
                    bulk_g2s_hint(ring_s + s * C::STAGE, c.src, c.nreal * C::TB, bar_s + 8 * s, pol);
                }
            } else {
                mbar_arrive(bar_s + 8 * s);
            }
        }
    };

    // The first stages of a dense launch are filled before the wait for the previous kernel: they
    // read only resident slot tiles, which no kernel that lets its dependents start early writes
    // (the store-side kernels run to completion before the next launch), so the first bytes
    // stream in while the previous merge finishes. Q, the suffix and the partials come after it.
    int inflight = 0;
    for (int s = 0; s < C::NSTAGE; ++s) {
        Chunk c;
        if (!cursor_next<FMT, D, C::TPS, C::TB>(p, prod, c)) break;
        issue(c, s);
        ++inflight;
    }
    if (!sparse) grid_dep_wait_then_release();

    StateT st;
    if constexpr (FMT == FMT_FP16) st.qsm = smem_u32(qarea);
    int cur_item = -1;
    int stage = 0;
    uint32_t phase = 0;
    Chunk c;
    while (cursor_next<FMT, D, C::TPS, C::TB>(p, cons, c)) {
        if (c.item != cur_item) {
            cur_item = c.item;
            if constexpr (FMT == FMT_FP16) start_item_f16<D, NCB>(st, p, p.desc[c.d], p.grp[c.grp], lane);
            else start_item_i4<D, NCB>(st, p, p.desc[c.d], p.grp[c.grp], lane);
        }
        if (!mbar_wait_bounded(bar_s + 8 * stage, (phase >> stage) & 1u)) {
            set_err(p.err, 1);
            for (int k = 1; k < inflight; ++k) {   // let the other copies land before leaving
                const int s2 = (stage + k) % C::NSTAGE;
                mbar_wait_bounded(bar_s + 8 * s2, (phase >> s2) & 1u);
            }
            return;
        }
        --inflight;
        const uint32_t head_mask = c.mask;   // bit h: local q head h attends to this chunk's tokens
        const uint8_t* sbuf = ring + stage * C::STAGE;
        for (int k = 0; k < c.nreal; ++k) {
            const int valid = c.valid - k * TILE_TOK, lo = c.lo - k * TILE_TOK;
            if constexpr (FMT == FMT_FP16) {
                const uint32_t sb = smem_u32(sbuf);
                SmemF16Tile<D> tl{sb + k * 32 * D, sb + C::STAGE / 2 + k * 32 * D, lane};
                tile_f16<D, NCB>(st, tl, lane, valid, head_mask, c.nq, lo);
            } else {
                if (D <= 128 && NCB == 1 && k + 3 < c.nreal) {   // four tiles per softmax step
                    tile_i4<D, NCB, 4>(st, sbuf + k * C::TB, lane, valid, head_mask, c.nq, lo);
                    k += 3;
                } else if (k + 1 < c.nreal) {   // two tiles per softmax step
                    tile_i4<D, NCB, 2>(st, sbuf + k * C::TB, lane, valid, head_mask, c.nq, lo);
                    ++k;
                } else {
                    tile_i4<D, NCB, 1>(st, sbuf + k * C::TB, lane, valid, head_mask, c.nq, lo);
                }
            }
        }
        phase ^= 1u << stage;
        __syncwarp();
        if (lane == 0) fence_proxy_async_smem();   // our reads of this stage precede the next copy into it
        Chunk nc;
        if (cursor_next<FMT, D, C::TPS, C::TB>(p, prod, nc)) {
            issue(nc, stage);
            ++inflight;
        }
        stage = stage + 1 == C::NSTAGE ? 0 : stage + 1;
        if (c.last) {
            if constexpr (FMT == FMT_FP16) finish_piece_f16<D, NCB>(st, p, cur_item, w + cur_item, lane);
            else finish_piece_i4<D, NCB>(st, p, cur_item, w + cur_item, lane);
            cur_item = -1;
        }
    }
}

template <int D, int NCB>
__device__ void suffix_worker(const DecodeParams& p, int sidx, int lane, uint8_t* qarea) {
    const int n_items = p.n_desc * p.n_groups;
    const int item = sidx / p.n_suf, k = sidx - item * p.n_suf;
    if (item >= n_items) return;
    const int d = item / p.n_groups, grp = item - d * p.n_groups;
    const DecodeDesc& ds = p.desc[d];
    const WorkGroup& wg = p.grp[grp];
    // The suffix is fp16 whatever the prefix format: fp16-style q fragments (no 1/16 factor).
    F16State<D, NCB> st;
    st.qsm = smem_u32(qarea);
    start_item_f16<D, NCB>(st, p, ds, wg, lane);
    const int t0 = 16 * k;
    GlobalF16Tile<D> tl{ds.Ksuf + (size_t)wg.g * p.S_suf * D, ds.Vsuf + (size_t)wg.g * p.S_suf * D, t0, p.S_suf, lane};
    tile_f16<D, NCB>(st, tl, lane, p.S_suf - t0, 0xFFFFFFFFu, wg.nq, ds.s_lo - t0);
    finish_piece_f16<D, NCB>(st, p, item, p.n_workers + n_items + item * p.n_suf + k, lane);
}

template <int FMT, int D, int NCB>
// An explicit minimum of one CTA per SM lifts ptxas's register budget for the int4 kernels (118
// registers at D=64, four CTAs per SM); fewer warps with more registers each measured faster than
// the higher occupancy of a tighter budget.
__global__ void __launch_bounds__(DECODE_WARPS * 32, 1) decode_kernel(const __grid_constant__ DecodeParams p) {
    using C = DCfg<FMT, D>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // worker ids go round the CTAs first, so that the prefix workers (and the suffix warps after
    // them) spread evenly over the SMs however many of them have work
    const int gw = warp * gridDim.x + blockIdx.x;
    uint8_t* ring = smem + warp * C::RING;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + DECODE_WARPS * C::RING) + warp * C::NSTAGE;
    uint8_t* qarea = smem + DECODE_WARPS * C::RING + DECODE_WARPS * C::NSTAGE * 8 + warp * C::QBYTES;
    if (gw < p.n_workers) {
        prefix_worker<FMT, D, NCB>(p, gw, lane, ring, bars, qarea);
    } else {
        grid_dep_wait_then_release();
        if (p.n_suf > 0) suffix_worker<D, NCB>(p, gw - p.n_workers, lane, qarea);
    }
}

// ---------------------------------------------------------------- host side

template <int FMT, int D, int NCB>
cudaError_t launch_t(const DecodeParams& p, int n_ctas, cudaStream_t st) {
    using C = DCfg<FMT, D>;
    static bool attr_set = false;   // per instantiation
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<FMT, D, NCB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t dc = {};
    dc.gridDim = dim3(n_ctas);
    dc.blockDim = dim3(DECODE_WARPS * 32);
    dc.dynamicSmemBytes = C::SMEM;
    dc.stream = st;
    dc.attrs = pdl;
    dc.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&dc, decode_kernel<FMT, D, NCB>, p);
    if (e != cudaSuccess) return e;
    // the merge of the partials, overlapping its launch with the decode's tail
    const int pairs = p.n_desc * p.n_groups * GMAX;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((pairs + 7) / 8);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, merge_kernel<D>, p);
}

template <int FMT, int D, int NCB>
DecodeLaunchInfo info_t() {
    using C = DCfg<FMT, D>;
    DecodeLaunchInfo i{C::STAGE, C::NSTAGE, C::SMEM, 0};
    int n = 0;
    cudaFuncSetAttribute(decode_kernel<FMT, D, NCB>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<FMT, D, NCB>, DECODE_WARPS * 32, C::SMEM) !=
        cudaSuccess)
        n = 1;
    i.ctas_per_sm = n > 0 ? n : 1;
    return i;
}

// Launch and occupancy of one (format, D) pair; instantiated by the translation units that own D.
// D = 512 has one column block only: its work groups hold at most 4 q heads.
template <int FMT, int D>
cudaError_t launch_d(const DecodeParams& p, int ncb, int n_ctas, cudaStream_t st) {
    if constexpr (D >= 512) return ncb == 1 ? launch_t<FMT, D, 1>(p, n_ctas, st) : cudaErrorInvalidValue;
    else return ncb == 1 ? launch_t<FMT, D, 1>(p, n_ctas, st) : launch_t<FMT, D, 2>(p, n_ctas, st);
}
template <int FMT, int D>
DecodeLaunchInfo info_d(int ncb) {
    if constexpr (D >= 512) return info_t<FMT, D, 1>();
    else return ncb == 1 ? info_t<FMT, D, 1>() : info_t<FMT, D, 2>();
}

}  // namespace pck
