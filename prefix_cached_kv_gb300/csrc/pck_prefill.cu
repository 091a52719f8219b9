// pck_prefill.cu -- batched-Q (M > 1) prefix attention on the 5th-generation tensor cores.
//
// "Shared KV Cache Serving -- Pion as LLM Memory", section "Wire-protocol details":
// ATTEND.PREFIX.QUERY with M query rows per head, Q of shape (H, M, D), answers with O and an
// LSE for every row;
// "ATTEND.* and ATTEND.PREFIX.*", section "Wire forms" / QUERY_FUSED: the prefix attention is
// merged with a dense suffix (here causal, bottom-right aligned: row i sees suffix keys
// j <= S_suf - M + i) in the same dispatch.
//
// One CTA owns 128 query rows of one kv head (the rows of its GQA q heads are packed:
// row = local head * M + i) and walks a contiguous range of that kv head's key blocks (64 keys;
// prefix then suffix); at D <= 128 two CTAs share an SM, so one's softmax runs while the other's
// MMAs do (at D = 256 the tile needs 512 TMEM columns and 192 KB of shared memory, one CTA per
// SM, and the next block's S = Q K^T overlaps the softmax instead):
//   * warp 5 (one lane) streams each block's K and V with cp.async.bulk into 2-stage K and V
//     rings (the resident fp16 layout already is the MMA operand layout);
//   * warp 4 issues tcgen05.mma (kind::f16, M=128, fp32 accumulators in TMEM) from one
//     elected lane: S = Q K^T into one of two S buffers (N = keys of the block, K-steps over
//     d), then O += P V with P read back from TMEM; S(b+1) runs while the softmax works on S(b);
//   * warps 0-3 (thread = row = TMEM lane) are the softmax: read S with tcgen05.ld, apply the
//     causal / length mask, write P = 2^(s - m) as packed fp16 over S and keep two running sums
//     (fp32 pairs through the packed f32x2 instructions): l_r of the fp16-rounded P, the
//     weights P.V actually multiplies, and l_x of the unrounded p; finally read O and write
//     O / l_r (a convex combination of the V rows whatever the rounding of P, so a large common
//     offset of V cancels exactly) and LSE = (m + log2 l_x) ln 2, or the partial of the key
//     range (merged by a second kernel).
// The running max m (base 2, tau*log2(e)-prescaled) is only moved when a 32-key chunk's sum
// exceeds 2^15 (which also bounds every P by 2^15, inside fp16): then O (in TMEM, once P.V of
// the previous block is done), l and the chunk are rescaled. Every wait is bounded: a stuck
// pipeline sets the device error word and the CTA still releases its tensor memory.
#include <math.h>

#include "pck_common.cuh"
#include "pck_kernels.h"

namespace pck {

namespace {

constexpr int PF_ROWS = 128;          // query rows per CTA (MMA M)
constexpr int PF_BLOCK = 64;          // keys per block (MMA N of S = Q K^T)
constexpr int PF_THREADS = 192;       // 4 softmax warps + MMA warp + producer warp
constexpr int PF_MMA_WARP = 4, PF_LOAD_WARP = 5;
constexpr int PF_ST = 2;              // K and V stages
constexpr float PF_LN2 = 0.69314718055994530942f;
// Launch-shape model of the key-range split, in units of one 64-key block of one CTA: a CTA's
// set-up and epilogue, and the merge kernel that a split adds.
constexpr double PF_CTA_COST = 2.0;
constexpr double PF_MERGE_COST = 4.0;

// Shared memory of one CTA: the Q tile and 2-stage K and V rings of 64-key blocks (two CTAs fit
// on an SM up to D = 128). Tensor memory: two S buffers (64 fp32 columns each; P of a block is
// written back over the first 32 columns of its buffer as packed fp16) and O (D columns).
template <int D>
struct PCfg {
    static constexpr int Q_BYTES = PF_ROWS * D * 2;
    static constexpr int KV_BYTES = PF_BLOCK * D * 2;         // K (or V) of one block
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + Q_BYTES;
    static constexpr int OFF_V = OFF_K + PF_ST * KV_BYTES;
    static constexpr int OFF_BAR = OFF_V + PF_ST * KV_BYTES;   // mbarriers + tmem slot
    static constexpr int SMEM = OFF_BAR + 256 + 128;           // + alignment slack (128 B)
    static constexpr int S_COL0 = 0, S_COL1 = PF_BLOCK;        // TMEM columns of the S buffers
    static constexpr int O_COL = 2 * PF_BLOCK;                 // TMEM columns of O (D)
    static constexpr int TMEM_COLS = O_COL + D <= 256 ? 256 : 512;   // a power of two
    static constexpr int CTAS_PER_SM = TMEM_COLS == 256 ? 2 : 1;     // TMEM holds 512 columns per SM
};

// ---------------------------------------------------------------- tcgen05 wrappers

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    // shared-memory matrix descriptor, no swizzle, K-major core matrices of 8 rows x 16 B
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;            // descriptor version for this architecture
    return d;                                        // base offset 0, layout type 0 (no swizzle)
}

__device__ __forceinline__ uint32_t idesc_f16(int M, int N) {
    // kind::f16: D f32, A/B f16, both K-major, no negation / sparsity
    return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// MMA (A and B from shared memory; or A from TMEM: row = lane, K packed two fp16 per 32-bit
// column) and commit, issued by one elected lane of a converged warp. The issuing warp runs
// its whole loop in step, so the descriptors stay warp-uniform values; computing them in
// lane-divergent code made each MMA issue cost about a hundred cycles.
__device__ __forceinline__ void umma_f16_elect(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{ .reg .pred p, e; .reg .b32 rx; elect.sync rx|e, 0xffffffff; setp.ne.u32 p, %4, 0; "
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }"
        ::"r"(tmem_d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

__device__ __forceinline__ void umma_f16_ts_elect(uint32_t tmem_d, uint32_t tmem_a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{ .reg .pred p, e; .reg .b32 rx; elect.sync rx|e, 0xffffffff; setp.ne.u32 p, %4, 0; "
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }"
        ::"r"(tmem_d), "r"(tmem_a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

__device__ __forceinline__ void umma_commit_elect(uint32_t bar) {
    asm volatile(
        "{ .reg .pred e; .reg .b32 rx; elect.sync rx|e, 0xffffffff; "
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0]; }"
        ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_st16_nowait(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
          "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// 16-column load, waited
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- softmax arithmetic

// two fp32 lanes in one 64-bit register (the packed f32x2 instructions of this architecture)
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
    uint64_t x;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a), "f"(b));
    return x;
}
__device__ __forceinline__ void f2_unpack(uint64_t x, float& a, float& b) { asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(x)); }
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// P of one 32-key chunk of a row: p_j = 2^(s_j sc - m) for the nv visible keys (0 for the
// rest), packed as fp16 pairs into pk; returns (sum of the fp16-rounded p_j, sum of the fp32 p_j).
template <bool FULL>
__device__ __forceinline__ float2 chunk_exp(const uint32_t (&v)[32], int lo, int nv, uint64_t sc2, float m,
                                            uint32_t (&pk)[16]) {
    const uint64_t nm2 = f2_pack(-m, -m);
    uint64_t ax0 = 0, ax1 = 0, ar0 = 0, ar1 = 0;   // (0.f, 0.f)
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1])), sc2, nm2), x0, x1);
        float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
        if (!FULL) {   // keys [lo, nv) of the chunk are visible
            p0 = 2 * j < nv && 2 * j >= lo ? p0 : 0.f;
            p1 = 2 * j + 1 < nv && 2 * j + 1 >= lo ? p1 : 0.f;
        }
        const __half2 h = __floats2half2_rn(p0, p1);
        const float2 r = __half22float2(h);
        if (j & 1) {
            ax1 = f2_add(ax1, f2_pack(p0, p1));
            ar1 = f2_add(ar1, f2_pack(r.x, r.y));
        } else {
            ax0 = f2_add(ax0, f2_pack(p0, p1));
            ar0 = f2_add(ar0, f2_pack(r.x, r.y));
        }
        pk[j] = h2_as_u32(h);
    }
    float a, b, c, d, e, f, g, k;
    f2_unpack(ax0, a, b);
    f2_unpack(ax1, c, d);
    f2_unpack(ar0, e, f);
    f2_unpack(ar1, g, k);
    return make_float2((e + f) + (g + k), (a + b) + (c + d));
}

// Sum of the 32 fp16 values packed in q.
__device__ __forceinline__ float half_sum32(const uint32_t (&q)[16]) {
    uint64_t a0 = 0, a1 = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const float2 r = __half22float2(u32_as_h2(q[j]));
        if (j & 1) a1 = f2_add(a1, f2_pack(r.x, r.y));
        else a0 = f2_add(a0, f2_pack(r.x, r.y));
    }
    float a, b, c, d;
    f2_unpack(a0, a, b);
    f2_unpack(a1, c, d);
    return (a + b) + (c + d);
}

// ---------------------------------------------------------------- work description

struct PfTask {
    int grp;        // work group (kv head + its q heads)
    int row0;       // first packed row of the CTA
};

struct PfParams {
    PrefillParams a;
    WorkGroup grp[MAX_GROUPS];
    int n_groups;
    int n_tiles;                    // row tiles over all groups
    int n_split;                    // key-range splits per row tile (CTAs = n_tiles * n_split)
    int task_off[MAX_GROUPS + 1];   // prefix sums of row tiles per group
    const uint8_t* suf_tiles;       // suffix in the resident fp16 layout (or nullptr)
    int suf_ntiles;
    float* partials;                // n_split > 1: [tile][split][row][partial_stride(D)]
};

// Key block b of a work unit's key sequence (row tile x key range): prefix blocks, then suffix.
struct KeyBlock {
    const uint8_t* k;
    const uint8_t* v;
    int ntile;       // resident 16-key tiles in the block
    int key0;        // first key index (within prefix or suffix)
    int is_suf;
};

__device__ __forceinline__ KeyBlock key_block(const PfParams& P, int g, int b, int nbp, int D) {
    KeyBlock kb;
    const int tiles_per_block = PF_BLOCK / TILE_TOK;
    if (b < nbp) {
        const size_t reg = fp16_region_bytes(P.a.ntiles, D);
        const uint8_t* base = P.a.kv + (size_t)g * 2 * reg;
        const int t0 = b * tiles_per_block;
        kb.ntile = min(tiles_per_block, P.a.ntiles - t0);
        kb.k = base + (size_t)t0 * 32 * D;
        kb.v = base + reg + (size_t)t0 * 32 * D;
        kb.key0 = t0 * TILE_TOK;
        kb.is_suf = 0;
    } else {
        const int bs = b - nbp;
        const size_t reg = fp16_region_bytes(P.suf_ntiles, D);
        const uint8_t* base = P.suf_tiles + (size_t)g * 2 * reg;
        const int t0 = bs * tiles_per_block;
        kb.ntile = min(tiles_per_block, P.suf_ntiles - t0);
        kb.k = base + (size_t)t0 * 32 * D;
        kb.v = base + reg + (size_t)t0 * 32 * D;
        kb.key0 = t0 * TILE_TOK;
        kb.is_suf = 1;
    }
    return kb;
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(PF_THREADS, 1) prefill_kernel(const __grid_constant__ PfParams P) {
    using C = PCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const uint32_t s_base = smem_u32(smem);
    // mbarriers (8 B each): K full / K free and V full / V free per stage, S full and P ready
    // (128 arrivals) per S buffer, P.V done, O final, drain. K(b) is released once S(b) is done,
    // V(b) once P(b).V is. No party can get a whole phase ahead of a waiter: the softmax arrives
    // P(b+2) only after S(b+2), which the issuer starts after it has seen P(b); the producer
    // refills a stage only after the issuer's commit for its previous contents.
    const uint32_t bar = s_base + C::OFF_BAR;
    constexpr int B_KF = 0, B_KE = 16, B_VF = 32, B_VE = 48, B_SF = 64, B_PR = 80, B_PV = 96, B_OF = 104,
                  B_DR = 112, N_BAR = 15;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 8 * N_BAR);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // the merge kernel (programmatic dependence) may be scheduled as this grid's CTAs retire; it
    // still waits for the whole grid before reading any partial
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // ---- which rows
    const int task = blockIdx.x / P.n_split;       // row tile
    const int split = blockIdx.x - task * P.n_split;
    int grp = 0;
    while (grp + 1 < P.n_groups && P.task_off[grp + 1] <= task) ++grp;
    const WorkGroup& wg = P.grp[grp];
    const int g = wg.g;
    const int M = P.a.M;
    const int rows_total = wg.nq * M;
    const int row0 = (task - P.task_off[grp]) * PF_ROWS;
    const int N = P.a.N, S = P.a.S_suf;
    const int nbp = (N + PF_BLOCK - 1) / PF_BLOCK;
    // suffix blocks needed by the last row of the tile (causal) or all of them
    int nbs = 0;
    if (S > 0) {
        int kmax = S;   // keys [0, kmax) of the suffix may be visible to some row of the tile
        if (P.a.causal) {
            const int last = min(rows_total, row0 + PF_ROWS) - 1;
            // rows are (local head, i): the largest i in the tile is M-1 if the tile crosses
            // the end of a head's rows, else that of its last row
            const int imax = (row0 / M != last / M) ? M - 1 : last % M;
            kmax = max(0, min(S, S - M + imax + 1));
        }
        nbs = (kmax + PF_BLOCK - 1) / PF_BLOCK;
    }
    const int nblocks = nbp + nbs;
    // this CTA's contiguous share of the key blocks (n_split <= nbp, so it is never empty)
    const int kb0 = static_cast<int>((static_cast<int64_t>(nblocks) * split) / P.n_split);
    const int kb1 = static_cast<int>((static_cast<int64_t>(nblocks) * (split + 1)) / P.n_split);
    const int nbl = kb1 - kb0;

    // ---- setup: barriers, TMEM, Q tile
    if (tid == 0) {
        for (int k = 0; k < N_BAR; ++k) mbar_init(bar + 8 * k, (8 * k == B_PR || 8 * k == B_PR + 8) ? 128 : 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_slot)), "r"(C::TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();   // barriers and the tensor-memory address visible to every warp
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // This grid may start before the previous kernel of the stream has finished (programmatic
    // dependence): the producer fetches the first stages of resident prefix blocks at once (no
    // kernel that releases its dependents early writes a slot's tiles, and a dequantised mlx4g32
    // copy is written by a kernel that runs to completion first); Q, the staged suffix and every
    // output wait for the previous grid.
    int pre = 0;   // stages issued before the wait (producer lane)
    if (warp == PF_LOAD_WARP && lane == 0) {
        for (; pre < PF_ST && pre < nbl && kb0 + pre < nbp; ++pre) {
            const KeyBlock kb = key_block(P, g, kb0 + pre, nbp, D);
            const uint32_t bytes = kb.ntile * 32 * D;
            mbar_arrive_expect_tx(bar + B_KF + 8 * pre, bytes);
            bulk_g2s(s_base + C::OFF_K + pre * C::KV_BYTES, kb.k, bytes, bar + B_KF + 8 * pre);
            mbar_arrive_expect_tx(bar + B_VF + 8 * pre, bytes);
            bulk_g2s(s_base + C::OFF_V + pre * C::KV_BYTES, kb.v, bytes, bar + B_VF + 8 * pre);
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (tid < PF_ROWS) {   // Q row -> core-matrix layout (zeros for rows past the end)
        const int r = row0 + tid;
        uint8_t* qs = smem + C::OFF_Q;
        const int R = tid >> 3, rr = tid & 7;
        if (r < rows_total) {
            const int h = wg.qh[r / M], i = r % M;
            const int qc = P.a.q_dup ? D / 16 : D / 8;   // 16-byte chunks of a source row
            const uint4* src = reinterpret_cast<const uint4*>(P.a.Q + ((size_t)h * M + i) * (qc * 8));
            // every 16-byte piece of the row in flight at once, straight into shared memory
            const uint32_t qs_s = smem_u32(qs);
#pragma unroll 8
            for (int c = 0; c < D / 8; ++c)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(qs_s + (R * (D / 8) + c) * 128 + rr * 16),
                             "l"(src + (c < qc ? c : c - qc)) : "memory");
            asm volatile("cp.async.commit_group;" ::: "memory");
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        } else {
#pragma unroll 4
            for (int c = 0; c < D / 8; ++c)
                *reinterpret_cast<uint4*>(qs + (R * (D / 8) + c) * 128 + rr * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    __syncthreads();   // the Q tile
    bool failed = false;

    if (warp == PF_LOAD_WARP) {
        // ------------------------------------------------------------ producer
        // One lane feeds both rings without blocking on either: K(j) needs S(j-2) done and V(j)
        // needs P(j-2).V done, and whichever stage frees first is refilled first (V never runs
        // ahead of K). Idle polls back off and are bounded like every other wait.
        if (lane == 0) {
            int jk = pre, jv = pre;
            uint32_t idle = 0;
            while (jv < nbl) {
                bool moved = false;
                if (jk < nbl && (jk < PF_ST || mbar_try_wait(bar + B_KE + 8 * (jk % PF_ST), (jk / PF_ST - 1) & 1))) {
                    const KeyBlock kb = key_block(P, g, kb0 + jk, nbp, D);
                    const uint32_t bytes = kb.ntile * 32 * D;
                    const int st = jk % PF_ST;
                    mbar_arrive_expect_tx(bar + B_KF + 8 * st, bytes);
                    bulk_g2s(s_base + C::OFF_K + st * C::KV_BYTES, kb.k, bytes, bar + B_KF + 8 * st);
                    ++jk;
                    moved = true;
                }
                if (jv < jk && (jv < PF_ST || mbar_try_wait(bar + B_VE + 8 * (jv % PF_ST), (jv / PF_ST - 1) & 1))) {
                    const KeyBlock kb = key_block(P, g, kb0 + jv, nbp, D);
                    const uint32_t bytes = kb.ntile * 32 * D;
                    const int st = jv % PF_ST;
                    mbar_arrive_expect_tx(bar + B_VF + 8 * st, bytes);
                    bulk_g2s(s_base + C::OFF_V + st * C::KV_BYTES, kb.v, bytes, bar + B_VF + 8 * st);
                    ++jv;
                    moved = true;
                }
                if (moved) {
                    idle = 0;
                } else {
                    if (++idle > (1u << 22)) { failed = true; break; }
                    if (idle > 64) __nanosleep(64);
                }
            }
            if (failed) set_err(P.a.err, 2);
        }
    } else if (warp == PF_MMA_WARP) {
        // ------------------------------------------------------------ MMA issuer
        // S(b) = Q K(b)^T into S buffer b%2; after the softmax has written P(b) over it,
        // O += P(b) V(b) with P read from tensor memory; S(b+2) reuses the buffer right after
        // (the MMAs of one thread execute in issue order), so S(b+1) overlaps softmax(b). The
        // whole warp walks the loop; lane 0 (elected) issues. Descriptors are built once and
        // advanced by adds (the start address field counts 16-byte units).
        const uint32_t o_tm = tmem + C::O_COL;
        const uint64_t q_desc = sdesc(s_base + C::OFF_Q, 128, 16 * D);
        const uint64_t k_desc = sdesc(s_base + C::OFF_K, 128, 16 * D);
        const uint64_t v_desc = sdesc(s_base + C::OFF_V, 128, 256);
        const uint32_t idesc_pv = idesc_f16(PF_ROWS, D);
        constexpr int TPB = PF_BLOCK / TILE_TOK;
        auto ntile_of = [&](int bi) -> int {
            const int b = kb0 + bi;
            return b < nbp ? min(TPB, P.a.ntiles - b * TPB) : min(TPB, P.suf_ntiles - (b - nbp) * TPB);
        };
        auto issue_S = [&](int bi) -> bool {
            const int st = bi % PF_ST;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar + B_KF + 8 * st, (bi / PF_ST) & 1))) return false;
            const uint32_t idesc = idesc_f16(PF_ROWS, ntile_of(bi) * TILE_TOK);
            const uint64_t kd = k_desc + static_cast<uint64_t>((st * C::KV_BYTES) >> 4);
            const uint32_t s_tm = tmem + ((bi & 1) ? C::S_COL1 : C::S_COL0);
#pragma unroll
            for (int s2 = 0; s2 < D / 16; ++s2) umma_f16_elect(s_tm, q_desc + 16 * s2, kd + 16 * s2, idesc, s2 > 0 ? 1u : 0u);
            umma_commit_elect(bar + B_SF + 8 * (bi & 1));   // S ready for the softmax
            umma_commit_elect(bar + B_KE + 8 * st);         // K stage free
            return true;
        };
        if (nbl > 0 && !issue_S(0)) failed = true;
        if (!failed && nbl > 1 && !issue_S(1)) failed = true;
        for (int bi = 0; bi < nbl && !failed; ++bi) {
            const int st = bi % PF_ST;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar + B_PR + 8 * (bi & 1), (bi >> 1) & 1) &&   // P(bi) written
                                             mbar_wait_bounded(bar + B_VF + 8 * st, (bi / PF_ST) & 1))) {
                failed = true;
                break;
            }
            tc_fence_after();
            const int nt = ntile_of(bi);
            const uint64_t vd = v_desc + static_cast<uint64_t>((st * C::KV_BYTES) >> 4);
            const uint32_t p_tm = tmem + ((bi & 1) ? C::S_COL1 : C::S_COL0);
#pragma unroll
            for (int u = 0; u < TPB; ++u)   // 16 keys (8 TMEM columns of P) per step
                if (u < nt) umma_f16_ts_elect(o_tm, p_tm + 8 * u, vd + ((u * 32 * D) >> 4), idesc_pv, (bi > 0 || u > 0) ? 1u : 0u);
            umma_commit_elect(bar + B_VE + 8 * st);   // V stage free once these complete
            umma_commit_elect(bar + B_PV);            // P.V of block bi done
            if (bi + 2 < nbl && !issue_S(bi + 2)) { failed = true; break; }
        }
        umma_commit_elect(bar + B_OF);                // O final (all earlier MMAs)
        if (failed && lane == 0) set_err(P.a.err, 3);
        // drain: make sure no MMA is still writing TMEM when the CTA releases it
        umma_commit_elect(bar + B_DR);
        __all_sync(0xffffffffu, mbar_wait_bounded(bar + B_DR, 0));
    } else {
        // ------------------------------------------------------------ softmax warps (row = tid)
        const int r = row0 + tid;
        const bool row_ok = r < rows_total;
        const int i = row_ok ? r % M : 0;
        const int suf_lim = P.a.causal ? (S - M + i) : (S - 1);   // last visible suffix key
        // first visible position of the prefix and suffix laid end to end (a window), else none
        const int first_pos = P.a.window > 0 ? N + S - M + i - P.a.window + 1 : -(1 << 30);
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        const uint32_t o_tm = tmem + C::O_COL + lane_base;
        const float sc = P.a.scale_log2;
        const uint64_t sc2 = f2_pack(sc, sc);
        float m = -INFINITY, lr = 0.f, lx = 0.f;   // running max; sums of rounded / exact P
        for (int bi = 0; bi < nbl; ++bi) {
            const uint32_t s_tm = tmem + ((bi & 1) ? C::S_COL1 : C::S_COL0) + lane_base;
            // warp-uniform outcome: the tcgen05.ld below must be executed by the whole warp
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar + B_SF + 8 * (bi & 1), (bi >> 1) & 1))) { failed = true; break; }
            tc_fence_after();
            const KeyBlock kb = key_block(P, g, kb0 + bi, nbp, D);
            const int ncols = kb.ntile * TILE_TOK;
            const int lim = kb.is_suf ? min(kb.key0 + ncols, suf_lim + 1) : min(kb.key0 + ncols, N);
            const int nvalid = row_ok ? max(0, lim - kb.key0) : 0;   // keys [key0, key0 + nvalid) visible
            const int nch = (ncols + 31) >> 5;
            uint32_t v[PF_BLOCK / 32][32];
#pragma unroll
            for (int c = 0; c < PF_BLOCK / 32; ++c)
                if (c < nch) tmem_ld32_nowait(s_tm + 32 * c, v[c]);
            tmem_wait_ld();
            float br = 0.f, bx = 0.f;   // this block's sums (rounded, exact) at the current m
#pragma unroll
            for (int c = 0; c < PF_BLOCK / 32; ++c) {
                if (c >= nch) break;
                const int nv = nvalid - 32 * c;   // visible keys of this chunk (<= 0 .. >= 32)
                // keys [lo, nv) of the chunk are visible: lo > 0 where a window starts inside it
                const int lo = max(0, first_pos - ((kb.is_suf ? N : 0) + kb.key0 + 32 * c));
                uint32_t pk[16];
                float2 cs = nv >= 32 && lo == 0 ? chunk_exp<true>(v[c], 0, nv, sc2, m, pk)
                                                : chunk_exp<false>(v[c], lo, nv, sc2, m, pk);
                // A sum <= 2^15 bounds every p_j by 2^15: they fit fp16 and m may stay. Otherwise
                // (or on the first chunk, where m = -inf and the sum is infinite) move m to the
                // chunk's max, rescale what was summed or written with the old m, and redo.
                const bool need = !(cs.y <= 32768.f);
                if (__any_sync(0xffffffffu, need)) {
                    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j < nv && j >= lo) mx[j & 3] = fmaxf(mx[j & 3], __uint_as_float(v[c][j]));
                    const float cm = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sc;
                    const float mnew = need ? fmaxf(m, cm) : m;
                    const float alpha = need ? exp2f(m - mnew) : 1.0f;
                    if (bi > 0) {   // O must be quiet: wait for P.V of the previous block
                        if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar + B_PV, (bi - 1) & 1))) { failed = true; break; }
                        tc_fence_after();
                        for (int c0 = 0; c0 < D; c0 += 16) {
                            uint32_t o[16];
                            tmem_ld16(o_tm + c0, o);
#pragma unroll
                            for (int j = 0; j < 16; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                            tmem_st16_nowait(o_tm + c0, o);
                        }
                    }
                    if (c > 0) {    // P of the earlier chunks, written over columns [0, 16c)
                        tmem_wait_st();
                        const __half2 a2 = __float2half2_rn(alpha);
                        br = 0.f;   // the rounded sum of what is stored after the rescale
                        for (int c1 = 0; c1 < c; ++c1) {
                            uint32_t q[16];
                            tmem_ld16(s_tm + 16 * c1, q);
#pragma unroll
                            for (int j = 0; j < 16; ++j) q[j] = h2_as_u32(__hmul2(u32_as_h2(q[j]), a2));
                            br += half_sum32(q);
                            tmem_st16_nowait(s_tm + 16 * c1, q);
                        }
                    }
                    tmem_wait_st();
                    bx *= alpha;
                    lr *= alpha;
                    lx *= alpha;
                    m = mnew;
                    cs = nv >= 32 && lo == 0 ? chunk_exp<true>(v[c], 0, nv, sc2, m, pk)
                                             : chunk_exp<false>(v[c], lo, nv, sc2, m, pk);
                }
                br += cs.x;
                bx += cs.y;
                // P of this chunk's 32 keys over columns [16c, 16c + 16): S there was read already
                tmem_st16_nowait(s_tm + 16 * c, pk);
            }
            if (failed) break;
            tmem_wait_st();
            lr += br;
            lx += bx;
            tc_fence_before();
            mbar_arrive(bar + B_PR + 8 * (bi & 1));
        }
        if (failed) {
            set_err(P.a.err, 4);
        } else if (__all_sync(0xffffffffu, mbar_wait_bounded(bar + B_OF, 0))) {
            tc_fence_after();
            // The row goes out through shared memory (the Q, K and V buffers are idle now that
            // every MMA has completed): the thread writes it there (a D + 4-word row
            // stride, so a quarter-warp's float4 stores hit 32 different banks) and sends it with
            // one bulk copy, instead of strided float4 stores to global memory.
            const bool fin = P.n_split == 1;
            const float inv = fin ? (lr > 0.f ? 1.0f / lr : 0.f) : 1.0f;
            constexpr int RS = partial_stride(D);   // floats per staged row
            float* srow = reinterpret_cast<float*>(smem) + (size_t)tid * RS;
            srow[0] = m;
            srow[1] = lr;
            srow[2] = lx;
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(o_tm + c0, v);
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4*>(srow + PARTIAL_O + c0 + j) =
                        make_float4(__uint_as_float(v[j]) * inv, __uint_as_float(v[j + 1]) * inv,
                                    __uint_as_float(v[j + 2]) * inv, __uint_as_float(v[j + 3]) * inv);
            }
            const int DO = P.a.q_dup ? D / 2 : D;   // columns of an output row
            if (fin && P.a.q_dup)
                for (int c = 0; c < D / 2; c += 4) {   // O = O_hi + O_lo
                    const float4 a = *reinterpret_cast<const float4*>(srow + PARTIAL_O + c);
                    const float4 b = *reinterpret_cast<const float4*>(srow + PARTIAL_O + D / 2 + c);
                    *reinterpret_cast<float4*>(srow + PARTIAL_O + c) = make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
                }
            if (row_ok) {
                fence_proxy_async_smem();   // this thread's writes, before its own bulk copy reads them
                if (fin) {   // O row, and LSE
                    bulk_s2g(P.a.O + ((size_t)wg.qh[r / M] * M + i) * DO, smem_u32(srow + PARTIAL_O), DO * 4);
                    if (P.a.LSE) P.a.LSE[(size_t)wg.qh[r / M] * M + i] = (m + log2f(lx)) * PF_LN2;
                } else {     // partial [m, l_r, l_x, -, o unnormalised] of this key range, merged later
                    bulk_s2g(P.partials + ((size_t)(task * P.n_split + split) * PF_ROWS + tid) * RS, smem_u32(srow),
                             RS * 4);
                }
                bulk_s2g_wait();
            }
        } else {
            set_err(P.a.err, 5);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS));
}

// Merge of the key-range partials of each row: one warp per row, lanes over d (float4; two of
// them per lane at D = 256). O is normalised by the merged sum of the rounded P, the LSE comes
// from the merged sum of the exact p (the two sums of the attention kernel). Small per-warp state
// (4 splits per batch) keeps many warps on an SM, so many rows' loads are in flight.
template <int D>
__global__ void __launch_bounds__(256) prefill_merge_kernel(const __grid_constant__ PfParams P) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int rows = P.n_tiles * PF_ROWS;
    constexpr int LPP = D / 4 < 32 ? D / 4 : 32;   // lanes holding the row's d
    constexpr int V4 = (D / 4 + LPP - 1) / LPP;      // float4 of d per lane
    for (int R = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; R < rows; R += (gridDim.x * blockDim.x) >> 5) {
        const int tile = R / PF_ROWS, rr = R - tile * PF_ROWS;
        int grp = 0;
        while (grp + 1 < P.n_groups && P.task_off[grp + 1] <= tile) ++grp;
        const WorkGroup& wg = P.grp[grp];
        const int M = P.a.M;
        const int r = (tile - P.task_off[grp]) * PF_ROWS + rr;
        if (r >= wg.nq * M) continue;
        const float* base = P.partials + ((size_t)tile * P.n_split * PF_ROWS + rr) * partial_stride(D);
        const size_t sstride = (size_t)PF_ROWS * partial_stride(D);
        // splits in batches of 4: a batch's (m, l_r, l_x) and o loads are all issued before any is used
        constexpr int NBS = 4;
        float Mx = -INFINITY, Lr = 0.f, Lx = 0.f;
        float4 acc[V4];
#pragma unroll
        for (int v = 0; v < V4; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c = 0; c < P.n_split; c += NBS) {
            const int nk = min(NBS, P.n_split - c);
            float4 ml = make_float4(-INFINITY, 0.f, 0.f, 0.f);
            if (lane < nk) ml = __ldcg(reinterpret_cast<const float4*>(base + (c + lane) * sstride));
            float4 xs[NBS][V4];
#pragma unroll
            for (int k = 0; k < NBS; ++k)
#pragma unroll
                for (int v = 0; v < V4; ++v)
                    xs[k][v] = (k < nk && lane < LPP && lane + v * LPP < D / 4)
                                   ? __ldcg(reinterpret_cast<const float4*>(base + (c + k) * sstride + PARTIAL_O) + lane + v * LPP)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
            float Mb = ml.x;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) Mb = fmaxf(Mb, __shfl_xor_sync(0xffffffffu, Mb, o));
            const float Mn = fmaxf(Mx, Mb);
            if (Mn != -INFINITY) {
                const float rs = Mx == -INFINITY ? 0.f : exp2f(Mx - Mn);   // rescale of earlier batches
                Lr *= rs;
                Lx *= rs;
#pragma unroll
                for (int v = 0; v < V4; ++v) { acc[v].x *= rs; acc[v].y *= rs; acc[v].z *= rs; acc[v].w *= rs; }
                Mx = Mn;
            }
            const float w = ml.x == -INFINITY ? 0.f : exp2f(ml.x - Mx);
            float Br = w * ml.y, Bx = w * ml.z;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                Br += __shfl_xor_sync(0xffffffffu, Br, o);
                Bx += __shfl_xor_sync(0xffffffffu, Bx, o);
            }
            Lr += Br;
            Lx += Bx;
#pragma unroll
            for (int k = 0; k < NBS; ++k) {
                const float ws = __shfl_sync(0xffffffffu, w, k);
#pragma unroll
                for (int v = 0; v < V4; ++v) {
                    acc[v].x = fmaf(ws, xs[k][v].x, acc[v].x); acc[v].y = fmaf(ws, xs[k][v].y, acc[v].y);
                    acc[v].z = fmaf(ws, xs[k][v].z, acc[v].z); acc[v].w = fmaf(ws, xs[k][v].w, acc[v].w);
                }
            }
        }
        const int h = wg.qh[r / M], i = r % M;
        const float inv = Lr > 0.f ? 1.0f / Lr : 0.f;
        if (!P.a.q_dup) {
            if (lane < LPP) {
#pragma unroll
                for (int v = 0; v < V4; ++v)
                    if (lane + v * LPP < D / 4)
                        reinterpret_cast<float4*>(P.a.O + ((size_t)h * M + i) * D)[lane + v * LPP] =
                            make_float4(acc[v].x * inv, acc[v].y * inv, acc[v].z * inv, acc[v].w * inv);
            }
        } else {   // O = O_hi + O_lo: float4 k and k + D/8 of the row
            float4* orow = reinterpret_cast<float4*>(P.a.O + ((size_t)h * M + i) * (D / 2));
            if constexpr (V4 == 2) {
                orow[lane] = make_float4((acc[0].x + acc[1].x) * inv, (acc[0].y + acc[1].y) * inv,
                                         (acc[0].z + acc[1].z) * inv, (acc[0].w + acc[1].w) * inv);
            } else {
                float4 b;
                b.x = __shfl_down_sync(0xffffffffu, acc[0].x, LPP / 2);
                b.y = __shfl_down_sync(0xffffffffu, acc[0].y, LPP / 2);
                b.z = __shfl_down_sync(0xffffffffu, acc[0].z, LPP / 2);
                b.w = __shfl_down_sync(0xffffffffu, acc[0].w, LPP / 2);
                if (lane < LPP / 2)
                    orow[lane] = make_float4((acc[0].x + b.x) * inv, (acc[0].y + b.y) * inv, (acc[0].z + b.z) * inv,
                                             (acc[0].w + b.w) * inv);
            }
        }
        if (lane == 0 && P.a.LSE) P.a.LSE[(size_t)h * M + i] = Lx > 0.f ? (Mx + log2f(Lx)) * PF_LN2 : -INFINITY;
    }
}

// The same merge when there are at most 4 splits (the usual case) and D <= 128: a warp takes 4
// consecutive rows of a tile and issues all of their loads (16 o float4 per lane, and lane
// 4q + k's (m, l_r, l_x) of row q, split k) before reducing any, so the whole merge is about one
// L2 round trip.
template <int D>
__global__ void __launch_bounds__(256, 3) prefill_merge4_kernel(const __grid_constant__ PfParams P) {
    static_assert(D <= 128, "four rows per warp hold D / 4 <= 32 lanes of o");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    constexpr int LPP = D / 4;   // lanes holding a row's d
    const int R0 = ((blockIdx.x * blockDim.x + threadIdx.x) >> 5) * 4;
    if (R0 >= P.n_tiles * PF_ROWS) return;
    const int tile = R0 / PF_ROWS, rr0 = R0 - tile * PF_ROWS;
    int grp = 0;
    while (grp + 1 < P.n_groups && P.task_off[grp + 1] <= tile) ++grp;
    const WorkGroup& wg = P.grp[grp];
    const int M = P.a.M, ns = P.n_split;
    const size_t sstride = (size_t)PF_ROWS * partial_stride(D);
    const float* base = P.partials + ((size_t)tile * ns * PF_ROWS + rr0) * partial_stride(D);
    const int mq = lane >> 2, mk = lane & 3;   // this lane's (row, split) for m, l_r and l_x
    float4 ml = make_float4(-INFINITY, 0.f, 0.f, 0.f);
    if (lane < 16 && mk < ns) ml = __ldcg(reinterpret_cast<const float4*>(base + mq * partial_stride(D) + mk * sstride));
    float4 xs[4][4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int k = 0; k < 4; ++k)
            xs[q][k] = (k < ns && lane < LPP)
                           ? __ldcg(reinterpret_cast<const float4*>(base + q * partial_stride(D) + k * sstride + PARTIAL_O) + lane)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
    // per row: max and the two sums over the lanes 4q .. 4q + 3
    float Mx = ml.x;
    Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, 1));
    Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, 2));
    const float w = ml.x == -INFINITY ? 0.f : exp2f(ml.x - Mx);
    float Lr = w * ml.y, Lx = w * ml.z;
    Lr += __shfl_xor_sync(0xffffffffu, Lr, 1);
    Lr += __shfl_xor_sync(0xffffffffu, Lr, 2);
    Lx += __shfl_xor_sync(0xffffffffu, Lx, 1);
    Lx += __shfl_xor_sync(0xffffffffu, Lx, 2);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float wk = __shfl_sync(0xffffffffu, w, 4 * q + k);
            acc.x = fmaf(wk, xs[q][k].x, acc.x); acc.y = fmaf(wk, xs[q][k].y, acc.y);
            acc.z = fmaf(wk, xs[q][k].z, acc.z); acc.w = fmaf(wk, xs[q][k].w, acc.w);
        }
        const float Lrq = __shfl_sync(0xffffffffu, Lr, 4 * q), Lxq = __shfl_sync(0xffffffffu, Lx, 4 * q);
        const float Mq = __shfl_sync(0xffffffffu, Mx, 4 * q);
        const int r = (tile - P.task_off[grp]) * PF_ROWS + rr0 + q;
        float4 b = make_float4(0.f, 0.f, 0.f, 0.f);   // q_dup: O_lo of this lane's columns
        if (P.a.q_dup) {
            b.x = __shfl_down_sync(0xffffffffu, acc.x, LPP / 2);
            b.y = __shfl_down_sync(0xffffffffu, acc.y, LPP / 2);
            b.z = __shfl_down_sync(0xffffffffu, acc.z, LPP / 2);
            b.w = __shfl_down_sync(0xffffffffu, acc.w, LPP / 2);
        }
        if (r >= wg.nq * M) continue;
        const int h = wg.qh[r / M], i = r % M;
        const float inv = Lrq > 0.f ? 1.0f / Lrq : 0.f;
        if (!P.a.q_dup) {
            if (lane < LPP)
                reinterpret_cast<float4*>(P.a.O + ((size_t)h * M + i) * D)[lane] =
                    make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        } else if (lane < LPP / 2) {
            reinterpret_cast<float4*>(P.a.O + ((size_t)h * M + i) * (D / 2))[lane] =
                make_float4((acc.x + b.x) * inv, (acc.y + b.y) * inv, (acc.z + b.z) * inv, (acc.w + b.w) * inv);
        }
        if (lane == 0 && P.a.LSE) P.a.LSE[(size_t)h * M + i] = Lxq > 0.f ? (Mq + log2f(Lxq)) * PF_LN2 : -INFINITY;
    }
}

bool prefill_supported(int D) {
    return D == 32 || D == 64 || D == 96 || D == 128 || D == 160 || D == 192 || D == 256;
}

template <int D>
static cudaError_t launch_prefill_t(const PfParams& P, cudaStream_t st) {
    using C = PCfg<D>;
    static_assert(C::CTAS_PER_SM * (C::SMEM + 1024) <= 233472, "the CTAs of an SM must fit its shared memory");
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    // Both launches are programmatic (PDL): the attention kernel may start while the suffix staging
    // runs (its prologue says what it reads before waiting), and the merge waits for the attention
    // grid as a whole.
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(P.n_tiles * P.n_split);
    cfg.blockDim = dim3(PF_THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = st;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, prefill_kernel<D>, P);
    if (e != cudaSuccess || P.n_split == 1) return e;
    const int rows = P.n_tiles * PF_ROWS;
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.numAttrs = 1;
    if constexpr (D <= 128) {
        if (P.n_split <= 4) {   // 4 rows per warp
            cfg.gridDim = dim3((rows + 31) / 32);
            return cudaLaunchKernelEx(&cfg, prefill_merge4_kernel<D>, P);
        }
    }
    cfg.gridDim = dim3((rows + 7) / 8);
    return cudaLaunchKernelEx(&cfg, prefill_merge_kernel<D>, P);
}

cudaError_t launch_prefill(const PrefillParams& a, const WorkGroup* grp, int n_groups, const void* suf_tiles,
                           int suf_ntiles, float* partials, size_t partial_bytes, int sms, cudaStream_t st, int D) {
    static thread_local PfParams P;
    P.a = a;
    P.n_groups = n_groups;
    int off = 0;
    for (int i = 0; i < n_groups; ++i) {
        P.grp[i] = grp[i];
        P.task_off[i] = off;
        off += (grp[i].nq * a.M + PF_ROWS - 1) / PF_ROWS;
    }
    P.task_off[n_groups] = off;
    P.n_tiles = off;
    P.suf_tiles = static_cast<const uint8_t*>(suf_tiles);
    P.suf_ntiles = suf_ntiles;
    P.partials = partials;
    if (off == 0) return cudaSuccess;
    // Key-range splits from a wave-cost model: with `slots` CTAs resident at once (two per SM up to
    // D = 128, one at D = 256), a launch of off * ns CTAs takes ceil(off * ns / slots) waves of
    // (nb / ns + PF_CTA_COST) block times, plus PF_MERGE_COST for the merge when ns > 1; never more
    // splits than prefix blocks, nor than the partials workspace holds.
    const int nbp = (a.N + PF_BLOCK - 1) / PF_BLOCK;
    const int nb = nbp + (a.S_suf + PF_BLOCK - 1) / PF_BLOCK;
    const int per_sm = D > 128 ? PCfg<256>::CTAS_PER_SM : PCfg<128>::CTAS_PER_SM;   // 512 TMEM columns above 128
    const int slots = per_sm * sms;
    int ns = 1;
    double best = 1e30;
    for (int k = 1; k <= 32 && k <= nbp; ++k) {
        if (static_cast<size_t>(off) * k * PF_ROWS * partial_stride(D) * sizeof(float) > partial_bytes) break;
        const double waves = static_cast<double>((static_cast<int64_t>(off) * k + slots - 1) / slots);
        const double cost = waves * (static_cast<double>(nb) / k + PF_CTA_COST) + (k > 1 ? PF_MERGE_COST : 0.0);
        if (cost < best - 1e-9) {
            best = cost;
            ns = k;
        }
    }
    P.n_split = ns;
    switch (D) {
        case 32: return launch_prefill_t<32>(P, st);
        case 64: return launch_prefill_t<64>(P, st);
        case 96: return launch_prefill_t<96>(P, st);
        case 128: return launch_prefill_t<128>(P, st);
        case 160: return launch_prefill_t<160>(P, st);
        case 192: return launch_prefill_t<192>(P, st);
        case 256: return launch_prefill_t<256>(P, st);
        default: break;
    }
    return cudaErrorInvalidValue;
}

}  // namespace pck
