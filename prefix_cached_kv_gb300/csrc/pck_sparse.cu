// pck_sparse.cu -- block-mean top-K selector feeding the sparse (gather) decode.
//
// "ATTEND.* and ATTEND.PREFIX.*", section "Wire forms" / QUERY_SPARSE_AUTO: the block means of K
// (block size B) are kept per slot; each q head's blocks are scored against its query and the
// K_top best are kept ("GQA-aware": a kv head's gather reads the union of its q heads' blocks
// once, each q head attending only to its own). Ties go to the lower block index; the
// selected indices are reported sorted ascending.
//
// Two kernels: score_kernel streams the block means through shared memory and writes every
// (q head, block) score; select_kernel (programmatic dependent launch) takes each q head's top-K,
// forms each work group's union of blocks with per-head masks, counts the resident tiles of the
// union (the gather decode's units) and, in the CTA that completes the last item, writes the
// items' unit offsets, from which the decode's workers split the selected tiles evenly.
#include <math.h>

#include <algorithm>

#include "pck_common.cuh"
#include "pck_kernels.h"
#include "pck_select.cuh"

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

// Split copy of the block means for the tensor-core scoring of the fused sparse kernel: one CTA
// per (group of 16 blocks, kv head); block r of the group and dimension d go to the core matrix
// (r / 8, d / 8) of the group's hi part (fp16(x)) and lo part (fp16(x - hi)), zeros past nb.
__global__ void __launch_bounds__(128) block_means_split_kernel(const float* __restrict__ kmean, int nb, int D,
                                                                uint8_t* __restrict__ out) {
    const int bg = blockIdx.x, g = blockIdx.y, nbg = gridDim.x;
    uint8_t* hi = out + ((size_t)g * nbg + bg) * 64 * D;
    uint8_t* lo = hi + 32 * D;
    for (int e = threadIdx.x; e < 16 * D; e += blockDim.x) {
        const int r = e / D, d = e - r * D, b = bg * 16 + r;
        const float x = b < nb ? kmean[((size_t)g * nb + b) * D + d] : 0.f;
        const __half h = __float2half_rn(x);
        const __half l = __float2half_rn(x - __half2float(h));
        const size_t off = ((size_t)(r >> 3) * (D / 8) + (d >> 3)) * 128 + (r & 7) * 16 + (d & 7) * 2;
        *reinterpret_cast<__half*>(hi + off) = h;
        *reinterpret_cast<__half*>(lo + off) = l;
    }
}

cudaError_t launch_block_means_split(const float* kmean, int H_kv, int nb, int D, uint8_t* out, cudaStream_t st) {
    if (D % 16 || nb < 1) return cudaErrorInvalidValue;
    block_means_split_kernel<<<dim3((nb + 15) / 16, H_kv), 128, 0, st>>>(kmean, nb, D, out);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- block scoring

// A scoring CTA takes a slab of SCORE_BPC consecutive blocks of one (session, kv head): one bulk
// copy brings the slab's block means (32 KB at D = 256) into shared memory, then each warp dots 8
// blocks with the kv head's q heads, 4 at a time, and sums the 8 x 4 per-lane products over the
// lanes by a reduce-scatter (31 shuffles for 32 sums; lane l ends with block l / 4, head l % 4):
// score[h, b] = tau * q_h . K_mean[head_map[h], b]. A kv head that no q head maps to scores
// nothing. The selection runs in its own grid (select_kernel, below).
constexpr int SEL_WARPS = 4;                           // warps per CTA (q heads taken in turn when selecting)
constexpr int SCORE_BPW = 8;                           // blocks per warp
constexpr int SCORE_BPC = SEL_WARPS * SCORE_BPW;       // blocks per CTA

template <int D>
__device__ __forceinline__ void score_blocks(const SelectParams& p, const SelSession& ss, int g, int b0, int nbl,
                                             const float* kslab, int lane) {
    constexpr int F4 = D / 4;                  // float4 per block mean
    constexpr int L4 = SCORE_BPW * F4 / 32;    // float4 per lane (16, 8, 4 for D = 256, 128, 64)
    constexpr int QN = F4 >= 32 ? F4 / 32 : 1; // float4 of one q head per lane
    // float4 e = lane + 32 k of the warp's blocks: block e / F4, float4 e % F4 of that block
    const float4* km = reinterpret_cast<const float4*>(kslab);
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
            const int e = lane + 32 * k;
            const float4 kv = e / F4 < nbl ? km[e] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 q = qv[j][F4 >= 32 ? k % QN : 0];
                float x = kv.x * q.x;
                x = fmaf(kv.y, q.y, x);
                x = fmaf(kv.z, q.z, x);
                x = fmaf(kv.w, q.w, x);
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

struct SelShared {
    int picks[GMAX][64];
    int sorted[GMAX][64];
    uint64_t cand[GMAX][32];
    uint8_t first[GMAX * 64];
    int scan[64];
    int cnt, last, nuniq;
};

// Selection for work group `grp` of session si, by a whole CTA (SEL_WARPS warps): warp w takes
// the top-K of the group's q heads w, w + SEL_WARPS, ... and sorts each ascending; then the CTA forms the group's
// sorted union of blocks, with a mask of the q heads that chose each, and the number of
// resident tiles the union covers (the item's units in the gather decode). The CTA that
// completes the last item of the launch turns the items' counts into their exclusive prefix
// (item_base), from which the decode's workers split the units evenly.
__device__ __forceinline__ void select_group(const SelectParams& p, int si, int grp, SelShared& sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const SelSession& ss = p.sess[si];
    const WorkGroup& wg = p.grp[grp];
    const int K = p.K_eff;
    if (threadIdx.x == 0) { sm.cnt = 0; sm.nuniq = 0; }
    for (int hw = warp; hw < wg.nq; hw += SEL_WARPS) {
        const int h = wg.qh[hw];
        const float* sc = ss.scores + (size_t)h * p.nb;
        constexpr int RPL = 32;                 // keys held in registers per lane (nb <= 1024)
        uint64_t key[RPL];
        const bool in_regs = p.nb <= 32 * RPL;
        if (in_regs) {
#pragma unroll
            for (int i = 0; i < RPL; ++i) {
                const int b = lane + 32 * i;
                key[i] = b < p.nb ? score_key(__ldcg(sc + b), b) : 0ull;
            }
        }
        const bool fast = in_regs && K <= 32 && topk_by_threshold(key, K, lane, sm.cand[hw], sm.picks[hw]);
        uint64_t prev = ~0ull;   // K rounds of arg-max below the previous pick
        for (int r = 0; r < (fast ? 0 : K); ++r) {
            uint64_t best = 0;
            if (in_regs) {
                uint64_t below[RPL];
#pragma unroll
                for (int i = 0; i < RPL; ++i) below[i] = key[i] < prev ? key[i] : 0ull;
                best = max32(below);
            } else {
                for (int b = lane; b < p.nb; b += 32) {
                    const uint64_t k = score_key(__ldcg(sc + b), b);
                    best = umax64(best, k < prev ? k : 0ull);
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) best = umax64(best, shfl64_xor(best, o));
            prev = best;
            if (lane == 0) sm.picks[hw][r] = key_block(best);
        }
        __syncwarp();
        // ascending order: a pick's place is the number of (distinct) picks below it
        for (int k = lane; k < K; k += 32) {
            const int v = sm.picks[hw][k];
            int r = 0;
            for (int j = 0; j < K; ++j) r += sm.picks[hw][j] < v ? 1 : 0;
            sm.sorted[hw][r] = v;
            if (ss.idx_out) ss.idx_out[(size_t)h * K + r] = v;
        }
    }
    __syncthreads();
    // union: entry (w, k) = head w's k-th smallest pick; the first head holding a block stands
    // for it. Lists are padded to 64 entries (index w * 64 + k, no divisions).
    const int nq = wg.nq;
    int nfirst = 0;
    for (int e = threadIdx.x; e < nq * 64; e += blockDim.x) {
        const int w = e >> 6, k = e & 63;
        bool f = false;
        if (k < K) {
            const int b = sm.sorted[w][k];
            f = true;
            for (int w2 = 0; w2 < w; ++w2)
                for (int k2 = 0; k2 < K; ++k2) f = f && sm.sorted[w2][k2] != b;
        }
        sm.first[e] = f ? 1 : 0;
        nfirst += f ? 1 : 0;
    }
    if (nfirst) atomicAdd(&sm.nuniq, nfirst);
    __syncthreads();
    const int nuniq = sm.nuniq;
    int* out_b = ss.sel_blocks + (size_t)grp * p.sel_max;
    uint8_t* out_m = ss.sel_mask + (size_t)grp * p.sel_max;
    for (int e = threadIdx.x; e < nq * 64; e += blockDim.x) {
        if (!sm.first[e]) continue;
        const int b = sm.sorted[e >> 6][e & 63];
        int rank = 0;   // distinct blocks below b
        uint32_t m = 0;
        for (int w2 = 0; w2 < nq; ++w2)
            for (int k2 = 0; k2 < K; ++k2) {
                const int v = sm.sorted[w2][k2];
                rank += (sm.first[w2 * 64 + k2] && v < b) ? 1 : 0;
                m |= (v == b ? 1u : 0u) << w2;
            }
        out_b[rank] = b;
        out_m[rank] = static_cast<uint8_t>(m);
        atomicAdd(&sm.cnt, min(p.tpb, p.ntiles - b * p.tpb));
    }
    for (int n = nuniq + threadIdx.x; n < p.sel_max; n += blockDim.x) { out_b[n] = -1; out_m[n] = 0; }
    __syncthreads();
    const int n_items = p.n_sess * p.n_groups;
    if (threadIdx.x == 0) {
        p.item_cnt[si * p.n_groups + grp] = sm.cnt;
        __threadfence();
        const unsigned old = atomicAdd(p.done, 1u);
        sm.last = old == static_cast<unsigned>(n_items) - 1u;
    }
    __syncthreads();
    if (!sm.last) return;
    __threadfence();
    // last item: exclusive prefix of the counts (a contiguous chunk per thread, then a block scan)
    const int nt = blockDim.x, per = (n_items + nt - 1) / nt;
    const int i0 = min(n_items, (int)threadIdx.x * per), i1 = min(n_items, i0 + per);
    int sum = 0;
    for (int i = i0; i < i1; ++i) sum += __ldcg(p.item_cnt + i);
    int x = sum;   // inclusive scan over the warp, then over the warps' totals
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sm.scan[warp] = x;
    __syncthreads();
    if (warp == 0) {
        const int nw = nt >> 5;
        int t = lane < nw ? sm.scan[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        if (lane < nw) sm.scan[32 + lane] = t;   // inclusive warp totals
        if (lane == nw - 1) {
            p.item_base[n_items] = t;
            *p.done = 0u;   // ready for the next launch
        }
    }
    __syncthreads();
    int run = x - sum + (warp > 0 ? sm.scan[32 + warp - 1] : 0);
    for (int i = i0; i < i1; ++i) {
        p.item_base[i] = run;
        run += __ldcg(p.item_cnt + i);
    }
}

// Scoring: one CTA of SEL_WARPS warps per slab (session, kv head, SCORE_BPC blocks): one bulk
// copy brings the slab's block means into shared memory, each warp scores 8 blocks. No atomics:
// a CTA leaves as soon as its scores are stored.
template <int D>
__global__ void __launch_bounds__(SEL_WARPS * 32, 4) score_kernel(const __grid_constant__ SelectParams p) {
    extern __shared__ __align__(128) uint8_t dsm[];   // the slab's block means, [SCORE_BPC][D] fp32
    __shared__ __align__(8) uint64_t bar;
    __shared__ int s_go;
    // the caller's inputs (and, for a first query, the block means) come from earlier kernels
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nbc = (p.nb + SCORE_BPC - 1) / SCORE_BPC;   // slabs per (session, kv head)
    const int per_sess = p.H_kv * nbc;
    const int si = blockIdx.x / per_sess, r = blockIdx.x - si * per_sess;
    const int g = r / nbc, b0 = (r - g * nbc) * SCORE_BPC;
    const int nbl = min(SCORE_BPC, p.nb - b0);
    const uint32_t bar_s = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(bar_s, 1);
        fence_mbar_init();
        const uint32_t bytes = static_cast<uint32_t>(nbl) * D * 4;
        mbar_arrive_expect_tx(bar_s, bytes);
        bulk_g2s(smem_u32(dsm), p.sess[si].kmean + ((size_t)g * p.nb + b0) * D, bytes, bar_s);
        s_go = mbar_wait_bounded(bar_s, 0) ? 1 : 0;
        if (!s_go) {
            set_err(p.err, 6);
            mbar_wait_bounded(bar_s, 0);   // let the copy land before the CTA leaves
        }
    }
    __syncthreads();
    // the select grid may launch once every CTA got here; it waits for this grid's completion
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int wb0 = warp * SCORE_BPW;
    if (s_go && wb0 < nbl)
        score_blocks<D>(p, p.sess[si], g, b0 + wb0, min(SCORE_BPW, nbl - wb0),
                        reinterpret_cast<const float*>(dsm) + (size_t)wb0 * D, lane);
}

// Selection: one CTA per (work group, session), after the scoring grid has completed.
__global__ void __launch_bounds__(SEL_WARPS * 32) select_kernel(const __grid_constant__ SelectParams p) {
    __shared__ SelShared sm;
    asm volatile("griddepcontrol.wait;" ::: "memory");   // every score is stored and visible
    // the decode grid may launch now; it waits for this grid's completion
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    select_group(p, blockIdx.y, blockIdx.x, sm);
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
    const int n_slabs = p.n_sess * p.H_kv * ((p.nb + SCORE_BPC - 1) / SCORE_BPC);
    const size_t smem = static_cast<size_t>(SCORE_BPC) * p.D * sizeof(float);
    void (*kern)(SelectParams) = p.D == 64 ? score_kernel<64> : p.D == 128 ? score_kernel<128>
                               : p.D == 256 ? score_kernel<256> : nullptr;
    if (!kern) return cudaErrorInvalidValue;
    static bool attr_set[3] = {false, false, false};
    const int ai = p.D == 64 ? 0 : p.D == 128 ? 1 : 2;
    if (!attr_set[ai]) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        attr_set[ai] = true;
    }
    // programmatic dependent launches: each grid's launch overlaps the previous kernel's tail,
    // and each kernel waits for that kernel's completion before reading anything
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t sc = {};
    sc.gridDim = dim3(static_cast<unsigned>(n_slabs));
    sc.blockDim = dim3(SEL_WARPS * 32);
    sc.dynamicSmemBytes = smem;
    sc.stream = st;
    sc.attrs = pdl;
    sc.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&sc, kern, p);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t sl = {};
    sl.gridDim = dim3(p.n_groups, p.n_sess);
    sl.blockDim = dim3(SEL_WARPS * 32);
    sl.stream = st;
    sl.attrs = pdl;
    sl.numAttrs = 1;
    return cudaLaunchKernelEx(&sl, select_kernel, p);
}

}  // namespace pck
