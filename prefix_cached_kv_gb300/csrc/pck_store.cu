// pck_store.cu -- store side: mlx4g32 quantiser and the re-layout of K/V into resident tiles.
//
// Quantiser: "Shared KV Cache Serving -- Pion as LLM Memory", section "Quantized tier --
// mlx4g32": 4-bit codes in groups of 32, affine with an fp16 scale and bias per group, codes
// picked against the fp16-rounded scale. A token's record is D/8 code words, D/32 fp16 scales,
// D/32 fp16 biases; a group's j-th code fills bits 4*(j mod 8) onward of its word.
#include "pck_common.cuh"
#include "pck_kernels.h"

namespace pck {

// ------------------------------------------------------------------ quantiser

template <typename SrcT>
__device__ __forceinline__ void load8(const SrcT* p, float (&x)[8]);

template <>
__device__ __forceinline__ void load8<__half>(const __half* p, float (&x)[8]) {
    uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __half22float2(h[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}

template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&x)[8]) {
    float4 a = __ldg(reinterpret_cast<const float4*>(p));
    float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// Codes of one word (8 elements) given its group's fp16 scale and bias, bit-exact with
// clamp(rint(fp32(fp32(x - bias) / scale)), 0, 15):
//   the quotient is first taken as a * RN(1/scale), which is within 2^-17 of the exact quotient
//   for |a/scale| <= 17 (two roundings of 2^-24 relative each); rint of it can only differ from
//   rint of the correctly rounded quotient when the value lies within 2^-16 of a half-integer,
//   and exactly those elements are redone with the IEEE division. Values far outside [0, 15]
//   clamp to the same code either way.
__device__ __forceinline__ uint32_t codes_of(const float (&x)[8], float sf, float bf, float rcp) {
    uint32_t w = 0;
    if (sf != 0.0f) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float a = __fsub_rn(x[k], bf);
            const float tp = __fmul_rn(a, rcp);
            float c = rintf(tp);
            if (fabsf(tp - c) > 0.5f - 1.52587890625e-05f) c = rintf(__fdiv_rn(a, sf));   // near a tie
            c = fminf(fmaxf(c, 0.0f), 15.0f);
            w |= static_cast<uint32_t>(c) << (4 * k);
        }
    }
    return w;
}

// One thread per pair of output code words (16 consecutive elements, 32 B of fp16 input); a group
// of 32 elements is 2 adjacent lanes. One pair per iteration with a register budget for six
// 256-thread CTAs per SM: more warps hide the load latency better than more loads per thread
// (measured: 107 us against 119 us for two pairs per iteration at four CTAs, 256 MB of input).
template <typename SrcT>
__global__ void __launch_bounds__(256, 6) quantize_mlx4g32_kernel(const SrcT* __restrict__ X, int64_t rows,
                                                                   int kv_dim, int lw, uint8_t* __restrict__ out) {
    // lw: log2 of the words per row when a power of two (a shift instead of a 64-bit division), else -1
    const int wpr = kv_dim / 8;                 // words per row
    const int64_t total = rows * wpr / 2;       // word pairs; even per group, a warp never splits one
    const int rec = kv_dim / 2 + kv_dim / 8;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t pi0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    // Every lane of a warp runs the same number of iterations, so the group shuffle below always
    // sees its partner (the 2 lanes of a group are both live or both idle).
    const int64_t iters = (total + stride - 1) / stride;
    for (int64_t it = 0; it < iters; ++it) {
        const int64_t pi = pi0 + it * stride;
        const bool live = pi < total;
        float x[2][8];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (live) {
                load8<SrcT>(X + (pi * 2 + h) * 8, x[h]);
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) x[h][k] = 0.f;
            }
        }
        float mn = x[0][0], mx = x[0][0];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int k = 0; k < 8; ++k) { mn = fminf(mn, x[h][k]); mx = fmaxf(mx, x[h][k]); }
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        const float s32 = __fdiv_rn(__fsub_rn(mx, mn), 15.0f);
        const __half s16 = __float2half_rn(s32);     // round-trip through fp16 first
        const __half b16 = __float2half_rn(mn);
        const float sf = __half2float(s16), bf = __half2float(b16);
        const float rcp = sf != 0.0f ? __frcp_rn(sf) : 0.0f;
        const uint32_t w0 = codes_of(x[0], sf, bf, rcp);
        const uint32_t w1 = codes_of(x[1], sf, bf, rcp);
        if (live) {
            const int64_t wi = pi * 2;
            const int64_t row = lw >= 0 ? wi >> lw : wi / wpr;
            const int word = static_cast<int>(wi - row * wpr);
            uint8_t* r = out + row * rec;
            reinterpret_cast<uint32_t*>(r)[word] = w0;        // records are only 4-byte aligned
            reinterpret_cast<uint32_t*>(r)[word + 1] = w1;
            if ((word & 3) == 0) {
                reinterpret_cast<__half*>(r + kv_dim / 2)[word >> 2] = s16;
                reinterpret_cast<__half*>(r + kv_dim / 2 + kv_dim / 16)[word >> 2] = b16;
            }
        }
    }
}

// ------------------------------------------------------------------ fp16 re-layout

// The 16 tokens of one tile, K and V rows of DS halves each, staged in shared memory (rows padded
// by 8 halves so that the column reads below spread over the banks) -> the tile's two 32*DS-byte
// pieces of the resident layout, written with consecutive 16-byte stores: the K piece as core
// matrices [token group][d chunk] (16 bytes = 8 consecutive d of one token), the V piece as core
// matrices [d group][key chunk] (16 bytes = 8 consecutive keys of one d).
template <int MAXD>
__device__ __forceinline__ void write_fp16_tile(const __half (&sm)[2][TILE_TOK][MAXD + 8], int DS, uint4* kout,
                                                uint4* vout) {
    const int piece = 2 * DS;                                 // uint4 per tile piece (32 * DS bytes)
    const int cpt = DS / 8;                                   // d chunks (K) / d groups (V)
    for (int u = threadIdx.x; u < piece; u += blockDim.x) {
        const int core = u >> 3, row = u & 7;
        const int T = core / cpt, c = core - T * cpt;         // K core: token group T, d chunk c
        kout[u] = *reinterpret_cast<const uint4*>(&sm[0][8 * T + row][8 * c]);
        const int dg = core >> 1, tc = core & 1, d = 8 * dg + row;   // V core: d group, key chunk
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = static_cast<uint32_t>(__half_as_ushort(sm[1][8 * tc + 2 * k][d])) |
                   (static_cast<uint32_t>(__half_as_ushort(sm[1][8 * tc + 2 * k + 1][d])) << 16);
        vout[u] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// One CTA per (16-token tile j, kv head g): K and V rows t0..t0+15 are loaded coalesced into
// shared memory (zeros past N), then written in the resident layout of head dimension DS >= D
// (columns D .. DS-1 zero: the [hi | lo] form of fp16 values, whose lo parts are 0). MAXD >= DS
// sizes the staging (256, or 512 for the widest heads, which halves the CTAs an SM holds).
// release: let the next kernel of the stream be scheduled at once (the batched-Q suffix staging,
// whose reader waits for this grid before it touches the staged suffix); the store path never
// does, so a slot's tiles are complete before any later kernel starts.
template <typename SrcT, int MAXD>
__global__ void __launch_bounds__(128) relayout_fp16_kernel(const SrcT* __restrict__ K, const SrcT* __restrict__ V,
                                                            int N, int D, int DS, int ntiles, uint4* __restrict__ out,
                                                            int release) {
    if (release) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ __align__(16) __half sm[2][TILE_TOK][MAXD + 8];
    const int j = blockIdx.x, g = blockIdx.y;
    const int t0 = j * TILE_TOK;
    for (int q = threadIdx.x; q < 2 * TILE_TOK * (DS - D) / 8; q += blockDim.x) {
        const int x = q / (TILE_TOK * (DS - D) / 8), r = q - x * (TILE_TOK * (DS - D) / 8);
        const int tok = r / ((DS - D) / 8), c = r - tok * ((DS - D) / 8);
        *reinterpret_cast<uint4*>(&sm[x][tok][D + 8 * c]) = make_uint4(0u, 0u, 0u, 0u);
    }
    for (int x = 0; x < 2; ++x) {
        const SrcT* src = (x ? V : K) + (int64_t)g * N * D;
        if constexpr (sizeof(SrcT) == 2) {
            for (int q = threadIdx.x; q < TILE_TOK * D / 8; q += blockDim.x) {
                const int tok = q / (D / 8), c = q - tok * (D / 8);
                uint4 val = make_uint4(0u, 0u, 0u, 0u);
                if (t0 + tok < N) val = __ldg(reinterpret_cast<const uint4*>(src + (int64_t)(t0 + tok) * D + 8 * c));
                *reinterpret_cast<uint4*>(&sm[x][tok][8 * c]) = val;
            }
        } else {
            for (int q = threadIdx.x; q < TILE_TOK * D; q += blockDim.x) {
                const int tok = q / D, d = q - tok * D;
                sm[x][tok][d] = __float2half_rn(t0 + tok < N ? static_cast<float>(src[(int64_t)(t0 + tok) * D + d]) : 0.f);
            }
        }
    }
    __syncthreads();
    const int64_t piece = 2 * DS;
    write_fp16_tile<MAXD>(sm, DS, out + ((int64_t)g * 2 * ntiles + j) * piece, out + ((int64_t)g * 2 * ntiles + ntiles + j) * piece);
}

// ------------------------------------------------------------------ QUERY_SPARSE token gather

// One CTA per (output tile j, q head h): the tokens idx[h][16j ..] (zeros past counts[h]) of kv
// head head_map[h] are read from the resident fp16 slot (K: 16 bytes of 8 d per token and d
// chunk; V: single values from the transposed tiles) into shared memory and written as tile j of
// head h's compact slot: K region of ceil(counts[h] / 16) tiles, then its V region, at
// out + h * head_stride bytes. MAXD >= D sizes the staging.
template <int MAXD>
__global__ void __launch_bounds__(128) gather_fp16_kernel(const uint8_t* __restrict__ tiles, int ntiles, int D,
                                                          const int* __restrict__ idx, const int* __restrict__ counts,
                                                          const int8_t* __restrict__ head_map, int kmax,
                                                          size_t head_stride, uint8_t* __restrict__ out) {
    __shared__ __align__(16) __half sm[2][TILE_TOK][MAXD + 8];
    const int j = blockIdx.x, h = blockIdx.y;
    const int cnt = counts[h];
    const int nt = (cnt + TILE_TOK - 1) / TILE_TOK;
    if (j >= nt) return;
    const int g = head_map[h];
    const uint8_t* kreg = tiles + (size_t)g * 2 * fp16_region_bytes(ntiles, D);
    const uint8_t* vreg = kreg + fp16_region_bytes(ntiles, D);
    const int* row = idx + (size_t)h * kmax;
    for (int q = threadIdx.x; q < TILE_TOK * D / 8; q += blockDim.x) {
        const int r = q / (D / 8), c = q - r * (D / 8);
        const int k = j * TILE_TOK + r;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (k < cnt) {
            const int t = row[k];
            val = __ldg(reinterpret_cast<const uint4*>(kreg + ((size_t)(t >> 3) * (D / 8) + c) * 128 + (t & 7) * 16));
        }
        *reinterpret_cast<uint4*>(&sm[0][r][8 * c]) = val;
    }
    for (int q = threadIdx.x; q < TILE_TOK * D; q += blockDim.x) {
        const int r = q / D, d = q - r * D;
        const int k = j * TILE_TOK + r;
        __half v = __float2half_rn(0.f);
        if (k < cnt) {
            const int t = row[k];
            v = *reinterpret_cast<const __half*>(vreg + (size_t)(t >> 4) * 32 * D + ((d >> 3) * 2 + ((t & 15) >> 3)) * 128 +
                                                 (d & 7) * 16 + (t & 7) * 2);
        }
        sm[1][r][d] = v;
    }
    __syncthreads();
    uint8_t* base = out + (size_t)h * head_stride;
    write_fp16_tile<MAXD>(sm, D, reinterpret_cast<uint4*>(base + (size_t)j * 32 * D),
                          reinterpret_cast<uint4*>(base + fp16_region_bytes(nt, D) + (size_t)j * 32 * D));
}

// ------------------------------------------------------------------ mlx4g32 tiles -> fp16 hi/lo pairs

// Code of (token tt, dimension d) of an mlx4g32 tile (layout in pck_common.cuh): K codes start at
// the tile, V codes at 10 * D bytes.
__device__ __forceinline__ uint32_t tile_k_code(const uint8_t* tile, int tt, int d) {
    const int s = d >> 4, w = d & 15, hi8 = w >> 3, q = (w & 7) >> 1, odd = w & 1;
    const int lane = 4 * (tt & 7) + q, n = (tt >> 3) + 2 * hi8 + 4 * odd;
    const uint32_t word = *reinterpret_cast<const uint32_t*>(tile + ((s >> 2) * 32 + lane) * 16 + (s & 3) * 4);
    return (word >> (4 * n)) & 0xFu;
}
__device__ __forceinline__ uint32_t tile_v_code(const uint8_t* vcodes, int tt, int d) {
    const int i = d >> 4, w = d & 15, dhi = w >> 3, t = w & 7;
    const int lane = 4 * t + ((tt & 7) >> 1), n = dhi + 2 * (tt >> 3) + 4 * (tt & 1);
    const uint32_t word = *reinterpret_cast<const uint32_t*>(vcodes + ((i >> 2) * 32 + lane) * 16 + (i & 3) * 4);
    return (word >> (4 * n)) & 0xFu;
}

// One CTA per (tile j, kv head g) of an mlx4g32 slot: every value x = scale * code + bias (fp32,
// one rounding) becomes an fp16 pair hi = fp16(x), lo = fp16(x - hi), and the tile is written as
// tile j of an fp16 slot of head dimension 2D whose first D columns are the hi parts and the
// last D the lo parts. Attention over that slot with Q' = [Q | Q] gives the scores of the
// dequantised K to ~22 bits, and P [V_hi | V_lo] gives O in two halves that sum to P V.
__global__ void __launch_bounds__(128) mlx4_tiles_split_kernel(const uint8_t* __restrict__ in, int ntiles, int D,
                                                               uint4* __restrict__ out) {
    constexpr int MAXD = 256;   // of the output (2D)
    __shared__ __align__(16) __half sm[2][TILE_TOK][MAXD + 8];
    __shared__ __align__(16) uint8_t tile[20 * (MAXD / 2)];   // the input tile (20 * D bytes)
    const int j = blockIdx.x, g = blockIdx.y;
    const uint4* src = reinterpret_cast<const uint4*>(in + ((size_t)g * ntiles + j) * tile_bytes(FMT_I4, D));
    for (int q = threadIdx.x; q < 20 * D / 16; q += blockDim.x) reinterpret_cast<uint4*>(tile)[q] = __ldg(src + q);
    __syncthreads();
    const int ng = D / 32;
    for (int q = threadIdx.x; q < 2 * TILE_TOK * D; q += blockDim.x) {
        const int x = q / (TILE_TOK * D), r = q - x * TILE_TOK * D;
        const int tt = r / D, d = r - tt * D;
        const uint32_t c = x ? tile_v_code(tile + 10 * D, tt, d) : tile_k_code(tile, tt, d);
        const __half2 sb = *reinterpret_cast<const __half2*>(tile + (x ? 18 : 8) * D + (tt * ng + (d >> 5)) * 4);
        const float v = fmaf(__low2float(sb), static_cast<float>(c), __high2float(sb));
        const __half hi = __float2half_rn(v);
        sm[x][tt][d] = hi;
        sm[x][tt][D + d] = __float2half_rn(v - __half2float(hi));
    }
    __syncthreads();
    const int64_t piece = 2 * (2 * D);
    write_fp16_tile<MAXD>(sm, 2 * D, out + ((int64_t)g * 2 * ntiles + j) * piece,
                          out + ((int64_t)g * 2 * ntiles + ntiles + j) * piece);
}

// ------------------------------------------------------------------ records -> [H_kv, N, D] (WARM)

// One thread per code word: 8 values of one token and one kv head, x = scale * code + bias in
// fp32 (one rounding of the exact value), stored at out[g][t][d0 .. d0 + 8) as fp32 or as the
// fp16 rounding of the fp32 value. Records are only 4-byte aligned (a record is kv_dim * 5/8 bytes).
template <typename OutT>
__global__ void __launch_bounds__(256) dequant_records_kernel(const uint8_t* __restrict__ rec, int64_t N, int H_kv,
                                                              int D, int lw, int lD, OutT* __restrict__ out) {
    // lw, lD: log2 of the words per record and of D when they are powers of two (shifts instead of
    // 64-bit divisions on every word), else -1
    const int kv_dim = H_kv * D, wpr = kv_dim / 8, rb = kv_dim / 2 + kv_dim / 8;
    const int64_t total = N * wpr;
    for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < total; w += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = lw >= 0 ? w >> lw : w / wpr;
        const int j = static_cast<int>(w - t * wpr);
        const uint8_t* r = rec + t * rb;
        const uint32_t word = __ldcs(reinterpret_cast<const uint32_t*>(r) + j);   // read once: streaming
        const int grp = j >> 2;   // 4 words per group of 32
        const float sc = __half2float(__ushort_as_half(__ldg(reinterpret_cast<const unsigned short*>(r + kv_dim / 2) + grp)));
        const float bi = __half2float(__ushort_as_half(__ldg(reinterpret_cast<const unsigned short*>(r + kv_dim / 2 + kv_dim / 16) + grp)));
        float x[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = fmaf(sc, static_cast<float>((word >> (4 * k)) & 0xFu), bi);
        const int e0 = 8 * j, g = lD >= 0 ? e0 >> lD : e0 / D, d0 = e0 - g * D;
        OutT* o = out + ((int64_t)g * N + t) * D + d0;
        // written once and not read back by this kernel: streaming (evict-first) stores
        if constexpr (sizeof(OutT) == 4) {
            __stcs(reinterpret_cast<float4*>(o), make_float4(x[0], x[1], x[2], x[3]));
            __stcs(reinterpret_cast<float4*>(o) + 1, make_float4(x[4], x[5], x[6], x[7]));
        } else {
            uint4 u;
            u.x = h2_as_u32(__floats2half2_rn(x[0], x[1]));
            u.y = h2_as_u32(__floats2half2_rn(x[2], x[3]));
            u.z = h2_as_u32(__floats2half2_rn(x[4], x[5]));
            u.w = h2_as_u32(__floats2half2_rn(x[6], x[7]));
            __stcs(reinterpret_cast<uint4*>(o), u);
        }
    }
}

// ------------------------------------------------------------------ mlx4g32 re-layout

struct RecSrc {
    const uint8_t* base;
    int head_rows;   // 1: rows are (g, t) with kv_dim = D; 0: rows are tokens with kv_dim = H_kv * D
    int H_kv, N, D;
};

__device__ __forceinline__ const uint8_t* rec_row(const RecSrc& s, int g, int t, int& kvr, int& goff) {
    if (s.head_rows) {
        kvr = s.D;
        goff = 0;
        return s.base + ((int64_t)g * s.N + t) * (s.D / 2 + s.D / 8);
    }
    kvr = s.H_kv * s.D;
    goff = g * s.D;
    return s.base + (int64_t)t * (kvr / 2 + kvr / 8);
}

__device__ __forceinline__ uint32_t rec_code(const RecSrc& s, int g, int t, int d) {
    if (t >= s.N) return 0;
    int kvr, goff;
    const uint8_t* r = rec_row(s, g, t, kvr, goff);
    const int e = goff + d;
    uint32_t w = reinterpret_cast<const uint32_t*>(r)[e >> 3];
    return (w >> (4 * (e & 7))) & 0xFu;
}

__device__ __forceinline__ uint32_t rec_sb(const RecSrc& s, int g, int t, int gi) {
    if (t >= s.N) return 0;
    int kvr, goff;
    const uint8_t* r = rec_row(s, g, t, kvr, goff);
    const int e = goff / 32 + gi;
    const uint16_t sc = reinterpret_cast<const uint16_t*>(r + kvr / 2)[e];
    const uint16_t bi = reinterpret_cast<const uint16_t*>(r + kvr / 2 + kvr / 16)[e];
    return static_cast<uint32_t>(sc) | (static_cast<uint32_t>(bi) << 16);
}

// One thread per output u32 of a tile (5 * D u32: K codes 2D, K sb D/2, V codes 2D, V sb D/2).
__global__ void __launch_bounds__(256) relayout_mlx4_kernel(RecSrc ks, RecSrc vs, int ntiles, uint32_t* __restrict__ out) {
    const int D = ks.D;
    const int words_tile = 5 * D;
    const int64_t total = (int64_t)ks.H_kv * ntiles * words_tile;
    const int ng = D / 32;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t tileg = i / words_tile;
        int w = static_cast<int>(i - tileg * words_tile);
        const int g = static_cast<int>(tileg / ntiles);
        const int j = static_cast<int>(tileg - (int64_t)g * ntiles);
        const int tb = j * TILE_TOK;
        bool isV = false;
        if (w >= 2 * D + D / 2) { isV = true; w -= 2 * D + D / 2; }
        const RecSrc& s = isV ? vs : ks;
        uint32_t val = 0;
        if (w < 2 * D) {                                 // codes word
            const int chunk = w / 128, lane = (w / 4) & 31, iw = chunk * 4 + (w & 3);
            const int q = lane & 3, l4 = lane >> 2;
            uint32_t nib[8];
            if (!isV) {   // K word iw = k-step s: the A fragment (tokens l4 and l4+8, d 16s + ...)
                const int s16 = 16 * iw;
                nib[0] = rec_code(s, g, tb + l4, s16 + 2 * q);
                nib[4] = rec_code(s, g, tb + l4, s16 + 2 * q + 1);
                nib[1] = rec_code(s, g, tb + 8 + l4, s16 + 2 * q);
                nib[5] = rec_code(s, g, tb + 8 + l4, s16 + 2 * q + 1);
                nib[2] = rec_code(s, g, tb + l4, s16 + 8 + 2 * q);
                nib[6] = rec_code(s, g, tb + l4, s16 + 9 + 2 * q);
                nib[3] = rec_code(s, g, tb + 8 + l4, s16 + 8 + 2 * q);
                nib[7] = rec_code(s, g, tb + 8 + l4, s16 + 9 + 2 * q);
            } else {   // V word iw = m-tile of d (16*iw ..): the A fragment of O^T = V^T P'^T
                const int d = 16 * iw + l4;
                nib[0] = rec_code(s, g, tb + 2 * q, d);
                nib[4] = rec_code(s, g, tb + 2 * q + 1, d);
                nib[1] = rec_code(s, g, tb + 2 * q, d + 8);
                nib[5] = rec_code(s, g, tb + 2 * q + 1, d + 8);
                nib[2] = rec_code(s, g, tb + 8 + 2 * q, d);
                nib[6] = rec_code(s, g, tb + 9 + 2 * q, d);
                nib[3] = rec_code(s, g, tb + 8 + 2 * q, d + 8);
                nib[7] = rec_code(s, g, tb + 9 + 2 * q, d + 8);
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) val |= nib[k] << (4 * k);
        } else {                                         // scale/bias word, [token][group]
            const int e = w - 2 * D;
            const int gi = e % ng, t = e / ng;
            val = rec_sb(s, g, tb + t, gi);
        }
        out[i] = val;
    }
}

// ------------------------------------------------------------------ host launchers

static int grid_for(int64_t work, int threads, int sms) {
    int64_t b = (work + threads - 1) / threads;
    int64_t cap = (int64_t)sms * 16;
    if (b > cap) b = cap;
    if (b < 1) b = 1;
    return static_cast<int>(b);
}

cudaError_t launch_quantize(const void* X, int src_f16, int64_t rows, int kv_dim, void* out, cudaStream_t st, int sms) {
    int64_t total = rows * (kv_dim / 16);   // word pairs
    int threads = 256;
    int blocks = grid_for(total, threads, sms);
    int lw = 0;
    while ((1 << lw) < kv_dim / 8) ++lw;
    if ((1 << lw) != kv_dim / 8) lw = -1;
    if (src_f16)
        quantize_mlx4g32_kernel<__half><<<blocks, threads, 0, st>>>(static_cast<const __half*>(X), rows, kv_dim, lw,
                                                                     static_cast<uint8_t*>(out));
    else
        quantize_mlx4g32_kernel<float><<<blocks, threads, 0, st>>>(static_cast<const float*>(X), rows, kv_dim, lw,
                                                                    static_cast<uint8_t*>(out));
    return cudaGetLastError();
}

cudaError_t launch_relayout_fp16(const void* K, const void* V, int src_f16, int H_kv, int N, int D, int ntiles,
                                 void* out, cudaStream_t st, int sms, int DS, int release) {
    (void)sms;
    if (DS == 0) DS = D;
    if (DS > 512 || D % 8 != 0 || DS % 8 != 0 || DS < D) return cudaErrorInvalidValue;
    const dim3 grid(ntiles, H_kv);
    const __half* kh = static_cast<const __half*>(K);
    const __half* vh = static_cast<const __half*>(V);
    const float* kf = static_cast<const float*>(K);
    const float* vf = static_cast<const float*>(V);
    uint4* o = static_cast<uint4*>(out);
    if (DS <= 256) {
        if (src_f16) relayout_fp16_kernel<__half, 256><<<grid, 128, 0, st>>>(kh, vh, N, D, DS, ntiles, o, release);
        else relayout_fp16_kernel<float, 256><<<grid, 128, 0, st>>>(kf, vf, N, D, DS, ntiles, o, release);
    } else {
        if (src_f16) relayout_fp16_kernel<__half, 512><<<grid, 128, 0, st>>>(kh, vh, N, D, DS, ntiles, o, release);
        else relayout_fp16_kernel<float, 512><<<grid, 128, 0, st>>>(kf, vf, N, D, DS, ntiles, o, release);
    }
    return cudaGetLastError();
}

cudaError_t launch_gather_fp16(const void* tiles, int ntiles, int D, const int* idx, const int* counts,
                               const int8_t* head_map, int H_q, int kmax, size_t head_stride, void* out, cudaStream_t st) {
    if (D > 512 || D % 16 != 0) return cudaErrorInvalidValue;
    const dim3 grid((kmax + TILE_TOK - 1) / TILE_TOK, H_q);
    const uint8_t* t = static_cast<const uint8_t*>(tiles);
    uint8_t* o = static_cast<uint8_t*>(out);
    if (D <= 256) gather_fp16_kernel<256><<<grid, 128, 0, st>>>(t, ntiles, D, idx, counts, head_map, kmax, head_stride, o);
    else gather_fp16_kernel<512><<<grid, 128, 0, st>>>(t, ntiles, D, idx, counts, head_map, kmax, head_stride, o);
    return cudaGetLastError();
}

cudaError_t launch_mlx4_split(const void* tiles, int H_kv, int ntiles, int D, void* out, cudaStream_t st) {
    if (2 * D > 256 || D % 32 != 0) return cudaErrorInvalidValue;
    const dim3 grid(ntiles, H_kv);
    mlx4_tiles_split_kernel<<<grid, 128, 0, st>>>(static_cast<const uint8_t*>(tiles), ntiles, D, static_cast<uint4*>(out));
    return cudaGetLastError();
}

cudaError_t launch_dequant_records(const void* rec, int64_t N, int H_kv, int D, int out_f16, void* out, cudaStream_t st,
                                   int sms) {
    const int64_t words = N * (H_kv * D / 8);
    const int blocks = grid_for(words, 256, sms);
    auto log2_exact = [](int v) {
        int l = 0;
        while ((1 << l) < v) ++l;
        return (1 << l) == v ? l : -1;
    };
    const int lw = log2_exact(H_kv * D / 8), lD = log2_exact(D);
    if (out_f16)
        dequant_records_kernel<__half><<<blocks, 256, 0, st>>>(static_cast<const uint8_t*>(rec), N, H_kv, D, lw, lD,
                                                                static_cast<__half*>(out));
    else
        dequant_records_kernel<float><<<blocks, 256, 0, st>>>(static_cast<const uint8_t*>(rec), N, H_kv, D, lw, lD,
                                                               static_cast<float*>(out));
    return cudaGetLastError();
}

cudaError_t launch_relayout_mlx4(const void* Krec, const void* Vrec, int head_rows, int H_kv, int N, int D, int ntiles,
                                 void* out, cudaStream_t st, int sms) {
    RecSrc ks{static_cast<const uint8_t*>(Krec), head_rows, H_kv, N, D};
    RecSrc vs{static_cast<const uint8_t*>(Vrec), head_rows, H_kv, N, D};
    int64_t total = (int64_t)H_kv * ntiles * 5 * D;
    int blocks = grid_for(total, 256, sms);
    relayout_mlx4_kernel<<<blocks, 256, 0, st>>>(ks, vs, ntiles, static_cast<uint32_t*>(out));
    return cudaGetLastError();
}

}  // namespace pck

// ------------------------------------------------------------------ host-buffer staging copy

namespace pck {

// One CTA per segment, 16-byte loads and stores; launched with programmatic dependence, it waits
// for the previous kernel of the stream before it overwrites the staging memory that kernel may
// still be reading.
__global__ void __launch_bounds__(256) copy_segments_kernel(const __grid_constant__ CopySegs p) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int sgi = blockIdx.x;
    if (sgi >= p.n) return;
    const uint4* src = static_cast<const uint4*>(p.src[sgi]);
    uint4* dst = static_cast<uint4*>(p.dst[sgi]);
    for (int i = threadIdx.x; i < p.n16[sgi]; i += blockDim.x) dst[i] = src[i];
}

cudaError_t launch_copy_segments(const CopySegs& p, cudaStream_t st) {
    if (p.n < 1 || p.n > MAX_COPY_SEGS) return cudaErrorInvalidValue;
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, copy_segments_kernel, p);
}

}  // namespace pck
