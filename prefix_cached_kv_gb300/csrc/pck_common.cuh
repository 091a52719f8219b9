// pck_common.cuh -- shared device helpers, resident tile layout and launch parameter blocks.
//
// Resident layout of a slot (one (sid, layer) of the ATTEND.PREFIX.STORE problem statement,
// "ATTEND.* and ATTEND.PREFIX.*", section "Wire forms"): per kv head g, the N prefix tokens are
// cut into 16-token tiles (the last one zero-padded).
//
//   FP16 slot: per kv head g, at base + g * ntiles * 64*D:
//     K region (ntiles * 32*D bytes): 8x8 "core matrices" of 8 tokens x 8 d (16 B per token row),
//        core (T, c) for token group T = t/8 and d chunk c = d/8 at (T * D/8 + c) * 128,
//        element (t, d) at row t%8 (16 B apart), halfword d%8.
//     V region (ntiles * 32*D bytes, right after K): per 16-token tile j, V transposed in core
//        matrices of 8 d x 8 tokens, core (dg, tc) for d group dg = d/8 and token chunk
//        tc = (t%16)/8 at j*32*D + (dg*2 + tc) * 128, element at row d%8, halfword t%8.
//     These are the no-swizzle K-major operand layouts of the tcgen05 MMA (S = Q K^T reads a
//     key block of any length with one descriptor, LBO = 128 B, SBO = 16*D B; O += P V reads
//     one 16-key tile per MMA, LBO = 128 B, SBO = 256 B), and word `lane` of a core matrix is
//     exactly the m16n8k16 B-fragment register of that lane, so the warp-MMA decode reads
//     its fragments with conflict-free 32-bit loads.
//
//   MLX4G32 tile (20*D bytes):  [K codes 8*D B][K sb 2*D B][V codes 8*D B][V sb 2*D B]
//     codes: lane l owns D/16 u32 words; word i at ((i/4)*32 + l)*16 + (i%4)*4; t = l/4, q = l%4.
//       K word s (k-step s, d = 16s..16s+15) is the lane's m16n8k16 A fragment with the 16
//       tokens of the tile as rows; nibble n (bits 4n..4n+3):
//           n0 = c[t][16s+2q]    n4 = c[t][16s+2q+1]    n1 = c[t+8][16s+2q]    n5 = c[t+8][16s+2q+1]
//           n2 = c[t][16s+8+2q]  n6 = c[t][16s+9+2q]    n3 = c[t+8][16s+8+2q]  n7 = c[t+8][16s+9+2q]
//       V word i (m-tile i, d = 16i + t): the lane's A fragment of O^T = V^T P'^T, d as rows:
//           n0 = c[2q][d]    n4 = c[2q+1][d]    n1 = c[2q][d+8]    n5 = c[2q+1][d+8]
//           n2 = c[8+2q][d]  n6 = c[9+2q][d]    n3 = c[8+2q][d+8]  n7 = c[9+2q][d+8]
//       so (w & 0x000F000F), (w & 0x00F000F0), ((w>>8) & 0x000F000F), ((w>>8) & 0x00F000F0) are
//       four half2 registers holding the codes as exact fp16 subnormals c * 2^-24 or 16c * 2^-24.
//     sb: [token 0..15][group 0..D/32) half2(scale, bias).
//
// The codes, scales and biases are the bytes of the mlx4g32 records ("Shared KV Cache Serving --
// Pion as LLM Memory", section "Quantized tier -- mlx4g32"), only permuted.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pck {

constexpr int FMT_FP16 = 0;
constexpr int FMT_I4 = 1;
constexpr int TILE_TOK = 16;       // tokens per resident tile
constexpr int GMAX = 8;            // q heads per work item (MMA rows 0-7 hi, 8-15 lo)
constexpr int MAX_DESC = 64;       // descriptors per launch
constexpr int MAX_GROUPS = 64;     // work groups (kv head x q-head batch)
constexpr int DECODE_WARPS = 4;    // warps per CTA (each an independent worker)

__host__ __device__ constexpr int tile_bytes(int fmt, int D) { return fmt == FMT_FP16 ? 64 * D : 20 * D; }
// Split-K partial of one q head: [m, l, pad, pad, o[0..D)] -- o starts 16-byte aligned.
__host__ __device__ constexpr int partial_stride(int D) { return D + 4; }
constexpr int PARTIAL_O = 4;   // float offset of o inside a head's partial
// fp16 slots: bytes of one kv head's K region (the V region follows it).
__host__ __device__ inline size_t fp16_region_bytes(int ntiles, int D) { return (size_t)ntiles * 32 * D; }

// ------------------------------------------------------------------ launch parameter blocks

struct DecodeDesc {
    const uint8_t* kv;      // resident tiles of this slot: [H_kv][ntiles][tile_bytes]
    const void* Q;          // [H_q, D] (q_f16 ? half : float)
    float* O;               // [H_q, D]
    float* LSE;             // [H_q] or nullptr
    const __half* Ksuf;     // [H_kv, S_suf, D] or nullptr
    const __half* Vsuf;
    const int* sel_blocks;  // sparse: [n_groups][sel_max] block ids (-1 = empty), or nullptr
    const uint8_t* sel_mask;// sparse: [n_groups][sel_max] bit h = local q head h selected it
    int N;                  // prefix tokens
    int ntiles;             // ceil(N / 16)
    int vtiles;             // tiles of one item's sequence (ntiles - tile0, or sel_max * tiles/block)
    int tile_off;           // first global tile of this descriptor's items
    // attention window (dense M=1): prefix tokens below t_lo and suffix tokens below s_lo are
    // masked; an item's tiles start at resident tile tile0 = t_lo / 16 (0 without a window)
    int t_lo, s_lo, tile0;
};

struct WorkGroup {
    int g;                  // kv head
    int nq;                 // q heads (<= GMAX)
    int8_t qh[GMAX];        // the q heads, local order
};

struct DecodeParams {
    DecodeDesc desc[MAX_DESC];
    WorkGroup grp[MAX_GROUPS];
    int n_desc, n_groups, H_q, H_kv, S_suf, q_f16;
    int total_tiles;        // dense: sum over items of vtiles
    int tpw;                // sparse: (unused) / dense: the target tiles per prefix worker
    // dense, aligned != 0: every item of descriptor d is cut into ppi[d] pieces of
    // ceil(vtiles / ppi[d]) tiles (the last one shorter), one per prefix worker; descriptor d's
    // workers start at wbase[d] (item (d, grp)'s pieces are workers wbase[d] + grp * ppi[d] ..),
    // wbase[n_desc] = n_workers. aligned == 0: worker w takes tiles [w tpw, (w+1) tpw) of the
    // items laid end to end (a range may straddle two items).
    int aligned;
    int ppi[MAX_DESC];
    int wbase[MAX_DESC + 1];
    int n_workers;          // prefix workers (warps)
    int n_suf;              // suffix pieces per item (ceil(S_suf / 16))
    int sparse;             // 1: item sequences come from sel_blocks
    int tiles_per_block;    // sparse: B / 16
    int sel_max;            // sparse: entries per group in sel_blocks
    int max_units;          // sparse: upper bound of the units of one launch (clamps item_base)
    const int* item_base;   // sparse: [n_items + 1] first unit (selected tile) of each item, written
                            // by the selector; the workers split [0, item_base[n_items]) evenly
    float scale_log2;       // tau * log2(e)
    float* partials;        // workspace: [slots][GMAX][partial_stride(D)]
    int* counters;          // workspace: [n_items]
    int* err;               // device error word (bounded waits that gave up)
};

// ------------------------------------------------------------------ small PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait on an mbarrier phase: gives up after ~2^22 polls (well over a second with the
// back-off) and returns false, so that a lost copy can never hang the GPU.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    for (uint32_t it = 0; it < (1u << 22); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (it > 64) __nanosleep(64);
    }
    return false;
}

// 1-D bulk copy shared -> global through the TMA engine (both addresses 16-byte aligned, bytes a
// multiple of 16), tracked by the issuing thread's bulk group; bulk_s2g_wait waits until the
// thread's copies are complete.
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes) : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_s2g_wait() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// 1-D bulk copy global -> shared through the TMA engine, completing on `bar` (tx bytes).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

// The same with an L2 eviction-priority hint (a policy from l2_evict_first()): for data read once
// per launch, so that it leaves L2 before what is read again (partials, q, suffixes).
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(pol) : "memory");
}
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// D(16x8 f32) += A(16x16 f16, row) * B(16x8 f16, col)
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// x -> (hi, lo) fp16 pair with hi + lo == x to ~22 bits; packs two values per register.
__device__ __forceinline__ void split_hi_lo(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    __half2 h = __floats2half2_rn(x0, x1);
    float2 hf = __half22float2(h);
    __half2 l = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
    hi = h2_as_u32(h);
    lo = h2_as_u32(l);
}

// The eight 4-bit codes of one word -> four half2 registers holding the codes as exact fp16
// subnormals: (w & 0x000F000F) is half2(c0 * 2^-24, c4 * 2^-24), (w & 0x00F000F0) is
// half2(16 c1 * 2^-24, 16 c5 * 2^-24), and the same on w >> 8 for c2, c6 / c3, c7. The tensor
// cores multiply subnormal fp16 inputs exactly; the 2^24 (or 2^20) goes into a later fp32 scale.
__device__ __forceinline__ void unpack_word(uint32_t w, uint32_t& p0, uint32_t& p1, uint32_t& p2, uint32_t& p3) {
    const uint32_t w8 = w >> 8;
    p0 = w & 0x000F000Fu;
    p1 = w & 0x00F000F0u;
    p2 = w8 & 0x000F000Fu;
    p3 = w8 & 0x00F000F0u;
}

// Transpose an 8x8 matrix of 16-bit values held in the m8n8 fragment layout (lane l: row l/4,
// columns 2(l%4), 2(l%4)+1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(x));
    return d;
}

// The hi and lo fp16 parts of two values, each pair in one register: a = half2(fp16(x0),
// fp16(x0 - fp16(x0))), b = the same for x1; the hi parts and the lo parts each take one paired
// conversion.
__device__ __forceinline__ void pack_hilo2(float x0, float x1, uint32_t& a, uint32_t& b) {
    const __half2 h = __floats2half2_rn(x0, x1);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
    const uint32_t hu = h2_as_u32(h), lu = h2_as_u32(l);
    a = __byte_perm(hu, lu, 0x5410);   // (hi0, lo0)
    b = __byte_perm(hu, lu, 0x7632);   // (hi1, lo1)
}

// 2^x with the hardware approximation (MUFU.EX2: ~2 ulp, flushes subnormal results to 0);
// used on base-2 scores that are <= 0 after the max subtraction, where its error is far below
// the 2e-3 / 1e-3 output tolerances.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void set_err(int* err, int code) {
    if (err) atomicCAS(err, 0, code);
}

}  // namespace pck
