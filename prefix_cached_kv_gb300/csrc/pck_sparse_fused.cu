// pck_sparse_fused.cu -- the block-mean top-K sparse query ("ATTEND.* and ATTEND.PREFIX.*",
// QUERY_SPARSE_AUTO(_FUSED)) as one kernel.
//
// One CTA per work item (session, group of q heads of one kv head g) runs every step of the
// query in shared memory:
//   1. scoring: each warp streams its own tiles of 16 block means (kept per slot as fp16 hi + lo
//      pairs, the same 4 bytes per value as fp32) through its own ring of bulk copies and scores
//      them on the tensor cores for every q head of the group; the scores
//      score[h, b] = tau * q_h . K_mean[g, b] stay in shared memory;
//   2. selection: warp w takes the top-K of q heads w, w + W, ... (ties to the lower block) and
//      marks them in a per-head map of blocks, from which the picks come out ascending and one
//      warp forms the union of the group's blocks with a mask of the q heads that chose each;
//   3. gather decode: the union's resident 16-token tiles and the dense suffix's 16-row tiles
//      (causal-free at M = 1; copied row-major, read by ldmatrix.trans for V) are split evenly
//      over the warps, each streaming its tiles through its own ring with the split-K decode's
//      tile step (each q head attends only to the blocks it chose);
//   4. merge: the warps' partials [m, l, o] are combined by their LSE and O, LSE written.
// Against the four-kernel form (scores, selection, gather decode, merge) this removes three
// kernel boundaries and the round trips of the scores and unit offsets through global memory.
// It needs the kv head's scores in shared memory (at most 1024 blocks) and K_top <= 64; larger
// cases take the four-kernel form.
#include "pck_decode_impl.cuh"
#include "pck_select.cuh"

namespace pck {

namespace {

constexpr int F_NBMAX = 1024;  // blocks per kv head whose scores fit in shared memory
constexpr int F_KMAX = 64;     // K_top limit

// Every warp streams its own copies: one warp's wait-and-reissue loop completes only a few
// bulk copies per microsecond, and one warp per scheduler leaves the tile math's dependent
// chains exposed, so a CTA runs as many warps as its rings fit in shared memory.
template <int D, int NCB>
struct FCfg {
    static constexpr int W = D == 256 ? 6 : 8;                 // warps per CTA
    static constexpr int HMAX = 4 * NCB;                       // q heads per group
    static constexpr int SLAB_BYTES = 64 * D;                  // a scoring stage: 16 blocks, hi and lo parts
    static constexpr int NSS = D == 64 ? 3 : 2;                // scoring stages per warp
    static constexpr int SCORE_RING = W * NSS * SLAB_BYTES;
    static constexpr int SCORES = HMAX * F_NBMAX * 4;
    static constexpr int TB = 64 * D;                          // fp16 tile: K 32 D bytes, then V 32 D bytes
    static constexpr int DST = D == 64 ? 4 : (D == 128 ? 3 : 2);   // decode ring stages per warp
    static constexpr int DRING = W * DST * TB;
    static constexpr int PART = W * HMAX * partial_stride(D) * 4;
    static constexpr int A1 = SCORE_RING + SCORES;
    static constexpr int REGION = A1 > DRING ? (A1 > PART ? A1 : PART) : (DRING > PART ? DRING : PART);
    static constexpr int NBAR = W * NSS + W * DST;
};

template <int HMAX>
struct FSel {
    int picks[HMAX][F_KMAX];
    uint64_t cand[HMAX][32];
    uint32_t bmap[HMAX][F_NBMAX / 32];   // each head's picks as a map of blocks
    int ublk[HMAX * F_KMAX];       // the union, ascending
    int utile[HMAX * F_KMAX + 1];  // exclusive prefix of the union's tiles
    uint8_t umask[HMAX * F_KMAX];
    int nuniq, fail;
};

template <int D, int NCB>
constexpr int fused_smem() {
    using C = FCfg<D, NCB>;
    return C::REGION + static_cast<int>(sizeof(FSel<C::HMAX>)) + C::NBAR * 8;
}

template <int D, int NCB>
__global__ void __launch_bounds__(FCfg<D, NCB>::W * 32, 1) sparse_fused_kernel(const __grid_constant__ FusedSparseParams p) {
    using C = FCfg<D, NCB>;
    constexpr int FW = C::W;
    constexpr int F_NSS = C::NSS;
    constexpr int HMAX = C::HMAX;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* regA = smem;
    FSel<HMAX>& sm = *reinterpret_cast<FSel<HMAX>*>(smem + C::REGION);
    const uint32_t bar0 = smem_u32(smem + C::REGION + sizeof(FSel<HMAX>));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int si = blockIdx.x / p.n_groups, grp = blockIdx.x - si * p.n_groups;
    const FusedSession& ss = p.sess[si];
    const WorkGroup& wg = p.grp[grp];
    const int g = wg.g, nq = wg.nq;
    auto sbar = [&](int s) { return bar0 + 8 * (warp * F_NSS + s); };
    auto dbar = [&](int s) { return bar0 + 8 * (FW * F_NSS + warp * C::DST + s); };
    if (tid == 0) {
        for (int k = 0; k < C::NBAR; ++k) mbar_init(bar0 + 8 * k, 1);
        fence_mbar_init();
        sm.fail = 0;
        sm.nuniq = 0;
    }
    __syncthreads();

    // ---------------------------------------------------------------- 1. scores
    // Each warp streams its own groups of 16 blocks (w, w + W, ...) of the split block means
    // through its own ring and scores them on the tensor cores, the blocks as MMA rows and the
    // q heads' hi / lo parts as columns: score = (K_hi + K_lo) . (q_hi + q_lo) tau, every product
    // exact and summed in fp32. The warps meet once every score is in shared memory.
    const int nb = p.nb;
    const int nbg = (nb + 15) / 16;
    const uint8_t* kmg = ss.kmean + (size_t)g * nbg * C::SLAB_BYTES;
    float* sc = reinterpret_cast<float*>(regA + C::SCORE_RING);   // [HMAX][F_NBMAX]
    uint8_t* sring = regA + warp * F_NSS * C::SLAB_BYTES;
    const uint32_t sring_s = smem_u32(sring);
    const uint64_t pol = l2_evict_first();   // block means and union tiles are read once per call
    auto issue_slab = [&](int j, int st) {   // the warp's j-th group (group w + j W) into stage st
        if (lane == 0) {
            mbar_arrive_expect_tx(sbar(st), C::SLAB_BYTES);
            bulk_g2s_hint(sring_s + st * C::SLAB_BYTES, kmg + (size_t)(warp + j * FW) * C::SLAB_BYTES, C::SLAB_BYTES, sbar(st), pol);
        }
    };
    const int mine = warp < nbg ? (nbg - warp + FW - 1) / FW : 0;   // groups of this warp
    for (int j = 0; j < min(F_NSS, mine); ++j) issue_slab(j, j);
    // The first stages above read only block means, which no kernel that lets its dependents start
    // early writes (they are built by kernels that run to completion); Q, the suffix and the
    // outputs may belong to the previous kernel of the stream, so wait for it from here on.
    grid_dep_wait_then_release();
    struct { int q_f16; float scale_log2; int* err; } qscale{p.q_f16, p.tau, p.err};
    F16State<D, NCB> sq;   // B fragments of tau * q (hi / lo parts), as the decode builds them
    sq.qsm = 0;
    start_item_f16<D, NCB>(sq, qscale, ss, wg, lane);
    for (int j = 0; j < mine; ++j) {
        const int st = j % F_NSS;
        if (!mbar_wait_bounded(sbar(st), (j / F_NSS) & 1)) {
            set_err(p.err, 6);
            sm.fail = 1;
            for (int k = j + 1; k < min(mine, j + F_NSS); ++k)   // let the other copies land first
                mbar_wait_bounded(sbar(k % F_NSS), (k / F_NSS) & 1);
            break;
        }
        const uint32_t sb = sring_s + st * C::SLAB_BYTES;
        const SmemF16Tile<D> thi{sb, 0u, lane}, tlo{sb + 32 * D, 0u, lane};
        float ah[NCB][4], al[NCB][4];
#pragma unroll
        for (int cb = 0; cb < NCB; ++cb)
#pragma unroll
            for (int i = 0; i < 4; ++i) ah[cb][i] = al[cb][i] = 0.f;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
            uint32_t a[4], b[4];
            thi.ka(k, a);
            tlo.ka(k, b);
#pragma unroll
            for (int cb = 0; cb < NCB; ++cb) {
                mma16816(ah[cb], a, sq.qb[cb][k][0], sq.qb[cb][k][1]);
                mma16816(al[cb], b, sq.qb[cb][k][0], sq.qb[cb][k][1]);
            }
        }
        const int b0 = (warp + j * FW) * 16 + (lane >> 2);
#pragma unroll
        for (int cb = 0; cb < NCB; ++cb) {
            const int hl = cb * 4 + (lane & 3);   // columns 2q, 2q + 1: head q's hi and lo parts
            if (hl < nq) {
                if (b0 < nb) sc[hl * F_NBMAX + b0] = (ah[cb][0] + al[cb][0]) + (ah[cb][1] + al[cb][1]);
                if (b0 + 8 < nb) sc[hl * F_NBMAX + b0 + 8] = (ah[cb][2] + al[cb][2]) + (ah[cb][3] + al[cb][3]);
            }
        }
        __syncwarp();
        if (j + F_NSS < mine) {
            if (lane == 0) fence_proxy_async_smem();   // the reads of this stage precede the next copy into it
            issue_slab(j + F_NSS, st);
        }
    }
    __syncthreads();
    if (sm.fail) return;

    // ---------------------------------------------------------------- 2. top-K and union
    // Each head's picks become a 1024-bit map of blocks (lane l: word l, blocks 32 l .. 32 l + 31):
    // the map read in lane order is the picks ascending, the OR of the maps is the union, a
    // block's bit in each map is its head mask, and ranks are popcounts under a warp scan.
    const int K = p.K_eff;
    for (int hw = warp; hw < nq; hw += FW) {
        const float* sch = sc + hw * F_NBMAX;
        uint64_t key[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int b = lane + 32 * i;
            key[i] = b < nb ? score_key(sch[b], b) : 0ull;
        }
        const bool fast = K <= 32 && topk_by_threshold(key, K, lane, sm.cand[hw], sm.picks[hw]);
        uint64_t prev = ~0ull;   // otherwise K rounds of arg-max below the previous pick
        for (int r = 0; r < (fast ? 0 : K); ++r) {
            uint64_t below[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) below[i] = key[i] < prev ? key[i] : 0ull;
            uint64_t best = max32(below);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) best = umax64(best, shfl64_xor(best, o));
            prev = best;
            if (lane == 0) sm.picks[hw][r] = key_block(best);
        }
        sm.bmap[hw][lane] = 0u;
        __syncwarp();
        for (int k = lane; k < K; k += 32) {
            const int v = sm.picks[hw][k];
            atomicOr(&sm.bmap[hw][v >> 5], 1u << (v & 31));
        }
        __syncwarp();
        // ascending picks: a block's place is the picks in lower words plus the lower bits of its own
        const uint32_t wbits = sm.bmap[hw][lane];
        const int cnt = __popc(wbits);
        int pre = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, pre, o);
            if (lane >= o) pre += y;
        }
        if (ss.idx_out) {
            const int h = wg.qh[hw];
            uint32_t m = wbits;
            for (int r = pre - cnt; m; ++r, m &= m - 1) ss.idx_out[(size_t)h * K + r] = 32 * lane + __ffs(m) - 1;
        }
    }
    __syncthreads();
    if (warp == 0) {   // the union, its head masks and its tiles' exclusive prefix, lane l over word l
        uint32_t u = 0;
        for (int w2 = 0; w2 < nq; ++w2) u |= sm.bmap[w2][lane];
        const int cnt = __popc(u);
        int tiles = 0;
        for (uint32_t m = u; m; m &= m - 1) {
            const int b = 32 * lane + __ffs(m) - 1;
            tiles += min(p.tpb, p.ntiles - b * p.tpb);
        }
        int pre = cnt, tpre = tiles;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, pre, o);
            const int z = __shfl_up_sync(0xffffffffu, tpre, o);
            if (lane >= o) { pre += y; tpre += z; }
        }
        int r = pre - cnt, run = tpre - tiles;
        for (uint32_t m = u; m; m &= m - 1, ++r) {
            const int bit = __ffs(m) - 1, b = 32 * lane + bit;
            uint32_t hm = 0;
            for (int w2 = 0; w2 < nq; ++w2) hm |= ((sm.bmap[w2][lane] >> bit) & 1u) << w2;
            sm.ublk[r] = b;
            sm.umask[r] = static_cast<uint8_t>(hm);
            sm.utile[r] = run;
            run += min(p.tpb, p.ntiles - b * p.tpb);
        }
        if (lane == 31) {
            sm.nuniq = pre;
            sm.utile[pre] = tpre;
        }
    }
    __syncthreads();
    const int nuniq = sm.nuniq;

    // ---------------------------------------------------------------- 3. gather decode
    const int upre = sm.utile[nuniq];
    const int n_suf = (p.S_suf + TILE_TOK - 1) / TILE_TOK;
    const int units = upre + n_suf;
    const int per_w = (units + FW - 1) / FW;
    const int u0 = min(units, warp * per_w), u1 = min(units, u0 + per_w);
    F16State<D, NCB> st;
    st.qsm = 0;
    start_item_f16<D, NCB>(st, p, ss, wg, lane);
    const size_t reg = fp16_region_bytes(p.ntiles, D);
    const uint8_t* kreg = ss.kv + (size_t)g * 2 * reg;
    const uint8_t* vreg = kreg + reg;
    uint8_t* ring = regA + warp * C::DST * C::TB;
    const uint32_t ring_s = smem_u32(ring);
    const int pe = u1;   // the warp's units are [u0, u1)
    // unit u -> (union entry, resident tile): entries are walked forward from the first one
    int ek = 0;
    {
        int lo = 0, hi = nuniq;   // the last entry whose first unit is <= u0
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (sm.utile[mid] <= u0) lo = mid; else hi = mid;
        }
        ek = lo;
    }
    int pk = ek;   // producer's entry
    auto tile_of = [&](int u, int& e) {
        while (e + 1 < nuniq && sm.utile[e + 1] <= u) ++e;
        return sm.ublk[e] * p.tpb + (u - sm.utile[e]);
    };
    // a unit below upre is a resident tile of the union; from upre on, 16 rows of the suffix,
    // copied row-major (a short last tile's missing rows are zeroed first, so that their zero
    // weights never meet stale bits)
    auto issue_tile = [&](int u, int s) {
        if (u < upre) {
            const int T = tile_of(u, pk);
            if (lane == 0) {
                mbar_arrive_expect_tx(dbar(s), C::TB);
                bulk_g2s_hint(ring_s + s * C::TB, kreg + (size_t)T * 32 * D, 32 * D, dbar(s), pol);
                bulk_g2s_hint(ring_s + s * C::TB + 32 * D, vreg + (size_t)T * 32 * D, 32 * D, dbar(s), pol);
            }
            return;
        }
        const int t0 = (u - upre) * TILE_TOK, rows = min(TILE_TOK, p.S_suf - t0);
        if (rows < TILE_TOK) {
            uint4* kz = reinterpret_cast<uint4*>(ring + s * C::TB + rows * 2 * D);
            uint4* vz = reinterpret_cast<uint4*>(ring + s * C::TB + 32 * D + rows * 2 * D);
            for (int i = lane; i < (TILE_TOK - rows) * D / 8; i += 32) {
                kz[i] = make_uint4(0u, 0u, 0u, 0u);
                vz[i] = make_uint4(0u, 0u, 0u, 0u);
            }
            __syncwarp();
        }
        if (lane == 0) {
            const uint32_t bytes = static_cast<uint32_t>(rows) * 2 * D;
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(dbar(s), 2 * bytes);
            bulk_g2s(ring_s + s * C::TB, ss.Ksuf + ((size_t)g * p.S_suf + t0) * D, bytes, dbar(s));
            bulk_g2s(ring_s + s * C::TB + 32 * D, ss.Vsuf + ((size_t)g * p.S_suf + t0) * D, bytes, dbar(s));
        }
    };
    // the rings reuse the memory of the scoring stages and the scores, which every warp has read
    // (generic proxy) before the last barrier: order those reads before the copies into it
    if (lane == 0) fence_proxy_async_smem();
    int next = u0, inflight = 0;
    for (int s = 0; s < C::DST && next < pe; ++s, ++next, ++inflight) issue_tile(next, s);
    uint32_t phase = 0;
    int stage = 0;
    for (int u = u0; u < pe; ++u) {
        const int T = u < upre ? tile_of(u, ek) : 0;
        if (!mbar_wait_bounded(dbar(stage), (phase >> stage) & 1u)) {
            set_err(p.err, 1);
            for (int k = 1; k < inflight; ++k) {   // let the other copies land before giving up
                const int s2 = (stage + k) % C::DST;
                mbar_wait_bounded(dbar(s2), (phase >> s2) & 1u);
            }
            break;
        }
        --inflight;
        const uint32_t sb = ring_s + stage * C::TB;
        if (u < upre) {
            SmemF16Tile<D> tl{sb, sb + 32 * D, lane};
            tile_f16<D, NCB>(st, tl, lane, min(TILE_TOK, p.N - T * TILE_TOK), sm.umask[ek], nq);
        } else {
            const int t0 = (u - upre) * TILE_TOK;
            SmemRowTile<D> tl{sb, sb + 32 * D, lane};
            tile_f16<D, NCB>(st, tl, lane, p.S_suf - t0, 0xFFFFFFFFu, nq);
        }
        phase ^= 1u << stage;
        __syncwarp();
        if (lane == 0) fence_proxy_async_smem();   // our reads of this stage precede the next copy into it
        if (next < pe) {
            issue_tile(next, stage);
            ++next;
            ++inflight;
        }
        stage = stage + 1 == C::DST ? 0 : stage + 1;
    }

    // ---------------------------------------------------------------- 4. merge of the warps' pieces
    __syncthreads();   // every ring is drained: the partials may overwrite them
    float* part = reinterpret_cast<float*>(regA);
    constexpr int PS = partial_stride(D);
    write_partial_f16<D, NCB>(st, part + warp * HMAX * PS, nq, lane);
    __syncthreads();
    constexpr int V = D / 32;   // o values per lane
    for (int hl = warp; hl < nq; hl += FW) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < FW; ++w) M = fmaxf(M, part[(w * HMAX + hl) * PS]);
        float L = 0.f, o[V];
#pragma unroll
        for (int v = 0; v < V; ++v) o[v] = 0.f;
#pragma unroll
        for (int w = 0; w < FW; ++w) {
            const float* ph = part + (w * HMAX + hl) * PS;
            const float mw = ph[0];
            const float wt = mw == -INFINITY ? 0.f : exp2f(mw - M);
            L = fmaf(wt, ph[1], L);
#pragma unroll
            for (int v = 0; v < V; ++v) o[v] = fmaf(wt, ph[PARTIAL_O + lane * V + v], o[v]);
        }
        const int qh = wg.qh[hl];
        const float inv = L > 0.f ? 1.0f / L : 0.f;
        float* orow = ss.O + (size_t)qh * D + lane * V;
#pragma unroll
        for (int v = 0; v < V; ++v) orow[v] = o[v] * inv;
        if (lane == 0 && ss.LSE) ss.LSE[qh] = L > 0.f ? (M + log2f(L)) * LN2 : -INFINITY;
    }
}

template <int D, int NCB>
cudaError_t launch_fused_t(const FusedSparseParams& p, cudaStream_t st) {
    constexpr int SMEM = fused_smem<D, NCB>();
    static_assert(SMEM <= 227 * 1024, "one CTA's shared memory");
    static bool attr = false;
    if (!attr) {
        const cudaError_t e = cudaFuncSetAttribute(sparse_fused_kernel<D, NCB>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.n_sess * p.n_groups));
    cfg.blockDim = dim3(FCfg<D, NCB>::W * 32);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, sparse_fused_kernel<D, NCB>, p);
}

}  // namespace

int sparse_fused_gmax(int D) { return D >= 256 ? 4 : GMAX; }

bool sparse_fused_ok(int D, int nb, int K_eff) {
    return (D == 64 || D == 128 || D == 256) && nb >= 1 && nb <= F_NBMAX && K_eff >= 1 && K_eff <= F_KMAX;
}

cudaError_t launch_sparse_fused(const FusedSparseParams& p, int max_nq, cudaStream_t st) {
    const int ncb = max_nq > 4 ? 2 : 1;
    if (p.D == 64) return ncb == 1 ? launch_fused_t<64, 1>(p, st) : launch_fused_t<64, 2>(p, st);
    if (p.D == 128) return ncb == 1 ? launch_fused_t<128, 1>(p, st) : launch_fused_t<128, 2>(p, st);
    if (p.D == 256 && ncb == 1) return launch_fused_t<256, 1>(p, st);
    return cudaErrorInvalidValue;
}

}  // namespace pck
