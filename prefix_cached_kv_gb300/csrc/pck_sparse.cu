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

// score[h, b] = tau * q_h . K_mean[head_map[h], b]; one warp per (session, kv head, 4 consecutive
// blocks): the 4 blocks' means are loaded together (32 loads per lane in flight at D = 256), then
// each q head of the kv head is read once and dotted with all 4.
constexpr int SCORE_BPW = 4;
__global__ void block_scores_kernel(const __grid_constant__ SelectParams p) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    const int nbw = (p.nb + SCORE_BPW - 1) / SCORE_BPW;   // warps per (session, kv head)
    const int per_sess = p.H_kv * nbw;
    if (warp >= p.n_sess * per_sess) return;
    const int si = warp / per_sess, wl = warp - si * per_sess;
    const SelSession& ss = p.sess[si];
    const int g = wl / nbw, b0 = (wl - g * nbw) * SCORE_BPW;
    const int per = p.D / 32;   // <= 8
    float kv[SCORE_BPW][8];
#pragma unroll
    for (int j = 0; j < SCORE_BPW; ++j) {
        const float* km = ss.kmean + ((size_t)g * p.nb + min(b0 + j, p.nb - 1)) * p.D;
#pragma unroll
        for (int i = 0; i < 8; ++i) kv[j][i] = i < per ? km[lane + 32 * i] : 0.f;
    }
    for (int h = 0; h < p.H_q; ++h) {
        if (p.head_map[h] != g) continue;
        float qv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int d = lane + 32 * i;
            qv[i] = i >= per ? 0.f
                             : (p.q_f16 ? __half2float(reinterpret_cast<const __half*>(ss.Q)[h * p.D + d])
                                        : reinterpret_cast<const float*>(ss.Q)[h * p.D + d]);
        }
#pragma unroll
        for (int j = 0; j < SCORE_BPW; ++j) {
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) acc = fmaf(qv[i], kv[j][i], acc);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0 && b0 + j < p.nb) ss.scores[(size_t)h * p.nb + b0 + j] = p.tau * acc;
        }
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

// One CTA per (work group, session): warp w selects the top-K of the group's w-th q head, then
// thread 0 merges the heads' selections into the group's sorted union (with per-head masks).
__global__ void select_kernel(const __grid_constant__ SelectParams p) {
    __shared__ int picks[GMAX][64];
    __shared__ float cand_s[GMAX][32];
    __shared__ int cand_i[GMAX][32];
    const int grp = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const SelSession& ss = p.sess[blockIdx.y];
    const WorkGroup& wg = p.grp[grp];
    const int K = p.K_eff;
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
        if (lane == 0) {   // ascending order
            for (int i = 1; i < K; ++i) {
                const int v = picks[warp][i];
                int j = i - 1;
                while (j >= 0 && picks[warp][j] > v) { picks[warp][j + 1] = picks[warp][j]; --j; }
                picks[warp][j + 1] = v;
            }
            if (ss.idx_out)
                for (int i = 0; i < K; ++i) ss.idx_out[(size_t)h * K + i] = picks[warp][i];
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int* out_b = ss.sel_blocks + (size_t)grp * p.sel_max;
        uint8_t* out_m = ss.sel_mask + (size_t)grp * p.sel_max;
        int pos[GMAX];
        for (int w = 0; w < wg.nq; ++w) pos[w] = 0;
        int n = 0;
        while (true) {   // k-way merge of the sorted per-head lists
            int best = 0x7fffffff;
            for (int w = 0; w < wg.nq; ++w)
                if (pos[w] < K && picks[w][pos[w]] < best) best = picks[w][pos[w]];
            if (best == 0x7fffffff) break;
            uint8_t m = 0;
            for (int w = 0; w < wg.nq; ++w)
                if (pos[w] < K && picks[w][pos[w]] == best) { m |= uint8_t(1u << w); ++pos[w]; }
            out_b[n] = best;
            out_m[n] = m;
            ++n;
        }
        for (; n < p.sel_max; ++n) { out_b[n] = -1; out_m[n] = 0; }
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
    block_scores_kernel<<<static_cast<unsigned>((warps + 7) / 8), 256, 0, st>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    select_kernel<<<dim3(p.n_groups, p.n_sess), GMAX * 32, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace pck
