// pck_sparse.cu -- block-mean top-K selector feeding the sparse (gather) decode.
//
// "ATTEND.* and ATTEND.PREFIX.*", section "Wire forms" / QUERY_SPARSE_AUTO: the block means of K
// (block size B) are kept per slot; each q head's blocks are scored against its query and the
// K_top best are kept ("GQA-aware": a kv head's gather reads the union of its q heads' blocks
// once, each q head attending only to its own). Ties go to the lower block index; the
// selected indices are reported sorted ascending.
#include <math.h>

#include "pck_common.cuh"
#include "pck_kernels.h"

namespace pck {

// K_mean[g, b, d] = mean over the tokens of block b of K[g, t, d] (fp32 sum of fp16 values),
// read from the K region of the resident fp16 slot (see pck_common.cuh).
__global__ void block_means_kernel(const uint8_t* __restrict__ tiles, int N, int D, int ntiles, int B,
                                   float* __restrict__ kmean) {
    const int b = blockIdx.x, g = blockIdx.y, nb = gridDim.x;
    const int t0 = b * B, t1 = min(N, t0 + B);
    const uint8_t* kreg = tiles + (size_t)g * 2 * fp16_region_bytes(ntiles, D);
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float acc = 0.f;
        for (int t = t0; t < t1; ++t) {
            const size_t off = ((size_t)(t >> 3) * (D / 8) + (d >> 3)) * 128 + (t & 7) * 16 + (d & 7) * 2;
            acc += __half2float(*reinterpret_cast<const __half*>(kreg + off));
        }
        kmean[((size_t)g * nb + b) * D + d] = acc / static_cast<float>(t1 - t0);
    }
}

// score[h, b] = tau * q_h . K_mean[head_map[h], b]. One warp per (session, kv head, 8 consecutive
// blocks): the 8 blocks' means (8 KB at D = 256) are read with 16-byte loads that are all in
// flight together, then dotted with the kv head's q heads, 4 at a time. The 8 x 4 per-lane dot
// products are summed over the lanes by a reduce-scatter (31 shuffles for 32 sums), after which
// lane l holds block l / 4 and head l % 4 of the batch.
constexpr int SCORE_BPW = 8;

template <int D>
__global__ void __launch_bounds__(128) block_scores_kernel(const __grid_constant__ SelectParams p) {
    constexpr int F4 = D / 4;                  // float4 per block mean
    constexpr int L4 = SCORE_BPW * F4 / 32;    // float4 per lane (16, 8, 4 for D = 256, 128, 64)
    constexpr int QN = F4 >= 32 ? F4 / 32 : 1; // float4 of one q head per lane
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    // the select launch that follows counts its finished CTAs from zero
    if (blockIdx.x == 0 && threadIdx.x == 0) *p.done = 0u;
    const int nbw = (p.nb + SCORE_BPW - 1) / SCORE_BPW;   // warps per (session, kv head)
    const int per_sess = p.H_kv * nbw;
    if (warp >= p.n_sess * per_sess) return;
    const int si = warp / per_sess, wl = warp - si * per_sess;
    const SelSession& ss = p.sess[si];
    const int g = wl / nbw, b0 = (wl - g * nbw) * SCORE_BPW;
    const int nbl = min(SCORE_BPW, p.nb - b0);
    // float4 e = lane + 32 k of the warp's blocks: block e / F4, float4 e % F4 of that block
    const float4* km = reinterpret_cast<const float4*>(ss.kmean + ((size_t)g * p.nb + b0) * D);
    float4 kv[L4];
#pragma unroll
    for (int k = 0; k < L4; ++k) {
        const int e = lane + 32 * k;
        kv[k] = e / F4 < nbl ? __ldg(km + e) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const int hb = lane + 32 < p.H_q ? p.head_map[lane + 32] : -1;
    const int ha = lane < p.H_q ? p.head_map[lane] : -1;
    uint64_t heads = (static_cast<uint64_t>(__ballot_sync(0xffffffffu, hb == g)) << 32) |
                     __ballot_sync(0xffffffffu, ha == g);
    while (heads) {
        int hh[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            hh[j] = heads ? __ffsll(static_cast<long long>(heads)) - 1 : -1;
            heads &= heads - 1;   // no-op once empty
        }
        float4 qv[4][QN];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int i = 0; i < QN; ++i) {
                const int d4 = F4 >= 32 ? lane + 32 * i : lane % F4;
                if (hh[j] < 0) {
                    qv[j][i] = make_float4(0.f, 0.f, 0.f, 0.f);
                } else if (p.q_f16) {
                    const uint2 r = __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const __half*>(ss.Q) + (size_t)hh[j] * D) + d4);
                    const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&r.x));
                    const float2 y = __half22float2(*reinterpret_cast<const __half2*>(&r.y));
                    qv[j][i] = make_float4(x.x, x.y, y.x, y.y);
                } else {
                    qv[j][i] = __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(ss.Q) + (size_t)hh[j] * D) + d4);
                }
            }
        }
        float acc[32];
#pragma unroll
        for (int v = 0; v < 32; ++v) acc[v] = 0.f;
#pragma unroll
        for (int k = 0; k < L4; ++k) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 q = qv[j][F4 >= 32 ? k % QN : 0];
                float x = kv[k].x * q.x;
                x = fmaf(kv[k].y, q.y, x);
                x = fmaf(kv[k].z, q.z, x);
                x = fmaf(kv[k].w, q.w, x);
                if constexpr (F4 >= 32) {
                    acc[(k / (F4 / 32)) * 4 + j] += x;
                } else {   // D = 64: lanes 0-15 hold block 2k, lanes 16-31 block 2k + 1
                    const bool hi = lane >= 16;
                    acc[(2 * k) * 4 + j] += hi ? 0.f : x;
                    acc[(2 * k + 1) * 4 + j] += hi ? x : 0.f;
                }
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {   // reduce-scatter: lane l ends with sum l
            const bool up = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < o; ++i) {
                const float send = up ? acc[i] : acc[i + o];
                const float keep = up ? acc[i + o] : acc[i];
                acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
        }
        const int blk = lane >> 2, j = lane & 3;
        const int h = j == 0 ? hh[0] : j == 1 ? hh[1] : j == 2 ? hh[2] : hh[3];
        if (h >= 0 && blk < nbl) ss.scores[(size_t)h * p.nb + b0 + blk] = p.tau * acc[0];
    }
}

__device__ __forceinline__ bool better(float sa, int ia, float sb, int ib) {
    return sa > sb || (sa == sb && ia < ib);
}

// Top-K of one q head's nb <= 1024 scores held 32 per lane (block b = lane + 32 i), when
// K <= 32: every lane finds its best element; the K-th best of those 32 lane bests, T, bounds
// the answer (the K lane bests ranked 0..K-1 are all at least T, so the K-th best score is too),
// so the top K are among the elements at least as good as T. When there are at most 32 of them
// they are gathered and each one's rank among them is its place; otherwise (many ties) the
// caller falls back to K rounds of arg-max. Order: higher score first, ties to the lower index.
__device__ __forceinline__ bool topk_by_threshold(const float (&reg)[32], int nb, int K, int lane, float* cs, int* ci,
                                                  int* picks) {
    constexpr int NONE = 0x7fffffff;
    float lb = -INFINITY;
    int li = NONE;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int b = lane + 32 * i;
        if (b < nb && (li == NONE || better(reg[i], b, lb, li))) { lb = reg[i]; li = b; }
    }
    int rank = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const float os = __shfl_sync(0xffffffffu, lb, j);
        const int oi = __shfl_sync(0xffffffffu, li, j);
        if (oi != NONE && (li == NONE || better(os, oi, lb, li))) ++rank;
    }
    const unsigned at = __ballot_sync(0xffffffffu, li != NONE && rank == K - 1);
    if (at == 0u) return false;
    const int src = __ffs(at) - 1;
    const float Ts = __shfl_sync(0xffffffffu, lb, src);
    const int Ti = __shfl_sync(0xffffffffu, li, src);
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int b = lane + 32 * i;
        cnt += (b < nb && (b == Ti || better(reg[i], b, Ts, Ti))) ? 1 : 0;
    }
    int pre = cnt;   // inclusive scan over lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, pre, o);
        if (lane >= o) pre += x;
    }
    const int C = __shfl_sync(0xffffffffu, pre, 31);
    if (C > 32) return false;
    int pos = pre - cnt;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int b = lane + 32 * i;
        if (b < nb && (b == Ti || better(reg[i], b, Ts, Ti))) { cs[pos] = reg[i]; ci[pos] = b; ++pos; }
    }
    __syncwarp();
    if (lane < C) {
        const float s = cs[lane];
        const int b = ci[lane];
        int r = 0;
        for (int k = 0; k < C; ++k) r += better(cs[k], ci[k], s, b) ? 1 : 0;
        if (r < K) picks[r] = b;
    }
    __syncwarp();
    return true;
}

// One CTA per (work group, session): warp w selects the top-K of the group's w-th q head and
// sorts it ascending; then the CTA forms the group's sorted union of blocks, with a mask of the
// q heads that chose each, and the number of resident tiles the union covers (the item's units
// in the gather decode). The last CTA of the launch to finish turns the items' counts into
// their exclusive prefix (item_base), from which the decode's workers split the units evenly.
__global__ void __launch_bounds__(GMAX * 32) select_kernel(const __grid_constant__ SelectParams p) {
    __shared__ int picks[GMAX][64];
    __shared__ int sorted[GMAX][64];
    __shared__ float cand_s[GMAX][32];
    __shared__ int cand_i[GMAX][32];
    __shared__ uint8_t first[GMAX * 64];
    __shared__ int s_cnt, s_last;
    __shared__ int s_scan[GMAX * 32];
    const int grp = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const SelSession& ss = p.sess[blockIdx.y];
    const WorkGroup& wg = p.grp[grp];
    const int K = p.K_eff;
    if (threadIdx.x == 0) s_cnt = 0;
    if (warp < wg.nq) {
        const int h = wg.qh[warp];
        const float* sc = ss.scores + (size_t)h * p.nb;
        constexpr int RPL = 32;                 // scores held in registers per lane (nb <= 1024)
        float reg[RPL];
        const bool in_regs = p.nb <= 32 * RPL;
        if (in_regs) {
#pragma unroll
            for (int i = 0; i < RPL; ++i) reg[i] = (lane + 32 * i < p.nb) ? sc[lane + 32 * i] : -INFINITY;
        }
        const bool fast = in_regs && K <= 32 && topk_by_threshold(reg, p.nb, K, lane, cand_s[warp], cand_i[warp], picks[warp]);
        float prev_s = INFINITY;
        int prev_i = -1;
        for (int r = 0; r < (fast ? 0 : K); ++r) {
            float bs = -INFINITY;
            int bi = 0x7fffffff;
            if (in_regs) {
#pragma unroll
                for (int i = 0; i < RPL; ++i) {
                    const int b = lane + 32 * i;
                    const float s = reg[i];
                    if (b < p.nb && better(prev_s, prev_i, s, b) && (bi == 0x7fffffff || better(s, b, bs, bi))) {
                        bs = s;
                        bi = b;
                    }
                }
            } else {
                for (int b = lane; b < p.nb; b += 32) {
                    const float s = sc[b];
                    if (better(prev_s, prev_i, s, b) && (bi == 0x7fffffff || better(s, b, bs, bi))) {
                        bs = s;
                        bi = b;
                    }
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float os = __shfl_xor_sync(0xffffffffu, bs, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (oi != 0x7fffffff && (bi == 0x7fffffff || better(os, oi, bs, bi))) {
                    bs = os;
                    bi = oi;
                }
            }
            prev_s = bs;
            prev_i = bi;
            if (lane == 0) picks[warp][r] = bi;
        }
        __syncwarp();
        // ascending order: a pick's place is the number of (distinct) picks below it
        for (int k = lane; k < K; k += 32) {
            const int v = picks[warp][k];
            int r = 0;
            for (int j = 0; j < K; ++j) r += picks[warp][j] < v ? 1 : 0;
            sorted[warp][r] = v;
            if (ss.idx_out) ss.idx_out[(size_t)h * K + r] = v;
        }
    }
    __syncthreads();
    // union: entry e = (head w, place k); the first head holding a block represents it
    const int ne = wg.nq * K;
    for (int e = threadIdx.x; e < ne; e += blockDim.x) {
        const int w = e / K, b = sorted[w][e - w * K];
        bool f = true;
        for (int w2 = 0; w2 < w; ++w2)
            for (int k = 0; k < K; ++k) f = f && sorted[w2][k] != b;
        first[e] = f ? 1 : 0;
    }
    __syncthreads();
    int* out_b = ss.sel_blocks + (size_t)grp * p.sel_max;
    uint8_t* out_m = ss.sel_mask + (size_t)grp * p.sel_max;
    int nuniq = 0;
    for (int e = 0; e < ne; ++e) nuniq += first[e];
    for (int e = threadIdx.x; e < ne; e += blockDim.x) {
        if (!first[e]) continue;
        const int w = e / K, b = sorted[w][e - w * K];
        int rank = 0;
        for (int e2 = 0; e2 < ne; ++e2) rank += (first[e2] && sorted[e2 / K][e2 % K] < b) ? 1 : 0;
        uint8_t m = 0;
        for (int w2 = 0; w2 < wg.nq; ++w2)
            for (int k = 0; k < K; ++k)
                if (sorted[w2][k] == b) m |= uint8_t(1u << w2);
        out_b[rank] = b;
        out_m[rank] = m;
        atomicAdd(&s_cnt, min(p.tpb, p.ntiles - b * p.tpb));
    }
    for (int n = nuniq + threadIdx.x; n < p.sel_max; n += blockDim.x) { out_b[n] = -1; out_m[n] = 0; }
    __syncthreads();
    const int n_items = p.n_sess * p.n_groups;
    if (threadIdx.x == 0) {
        p.item_cnt[blockIdx.y * p.n_groups + grp] = s_cnt;
        __threadfence();
        const unsigned old = atomicAdd(p.done, 1u);
        s_last = old == static_cast<unsigned>(n_items) - 1u;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // last CTA: exclusive prefix of the counts (a contiguous chunk per thread, then a block scan)
    const int nt = blockDim.x, per = (n_items + nt - 1) / nt;
    const int i0 = min(n_items, (int)threadIdx.x * per), i1 = min(n_items, i0 + per);
    int sum = 0;
    for (int i = i0; i < i1; ++i) sum += __ldcg(p.item_cnt + i);
    s_scan[threadIdx.x] = sum;
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int t = 0; t < nt; ++t) { const int x = s_scan[t]; s_scan[t] = run; run += x; }
        p.item_base[n_items] = run;
        *p.done = 0u;
    }
    __syncthreads();
    int run = s_scan[threadIdx.x];
    for (int i = i0; i < i1; ++i) {
        p.item_base[i] = run;
        run += __ldcg(p.item_cnt + i);
    }
}

cudaError_t launch_block_means(const void* tiles, int H_kv, int N, int D, int ntiles, int B, float* kmean,
                               cudaStream_t st, int sms) {
    (void)sms;
    const int nb = (N + B - 1) / B;
    dim3 grid(nb, H_kv);
    block_means_kernel<<<grid, D < 128 ? D : 128, 0, st>>>(static_cast<const uint8_t*>(tiles), N, D, ntiles, B, kmean);
    return cudaGetLastError();
}

cudaError_t launch_select(const SelectParams& p, cudaStream_t st, int sms) {
    (void)sms;
    const int64_t warps = static_cast<int64_t>(p.n_sess) * p.H_kv * ((p.nb + SCORE_BPW - 1) / SCORE_BPW);
    const unsigned ctas = static_cast<unsigned>((warps + 3) / 4);
    if (p.D == 64) block_scores_kernel<64><<<ctas, 128, 0, st>>>(p);
    else if (p.D == 128) block_scores_kernel<128><<<ctas, 128, 0, st>>>(p);
    else if (p.D == 256) block_scores_kernel<256><<<ctas, 128, 0, st>>>(p);
    else return cudaErrorInvalidValue;
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    select_kernel<<<dim3(p.n_groups, p.n_sess), GMAX * 32, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace pck
