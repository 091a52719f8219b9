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
                                                                   int kv_dim, uint8_t* __restrict__ out) {
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
            const int64_t row = wi / wpr;
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

// One CTA per (16-token tile j, kv head g). K and V rows t0..t0+15 are loaded coalesced into
// shared memory (zeros past N; rows padded by 16 bytes so the column reads below spread over
// the banks), then the tile's two 32*D-byte pieces of the resident layout are written with
// consecutive 16-byte stores: the K piece as core matrices [token group][d chunk] (16 bytes =
// 8 consecutive d of one token), the V piece as core matrices [d group][key chunk] (16 bytes =
// 8 consecutive keys of one d).
template <typename SrcT>
__global__ void __launch_bounds__(128) relayout_fp16_kernel(const SrcT* __restrict__ K, const SrcT* __restrict__ V,
                                                            int N, int D, int ntiles, uint4* __restrict__ out) {
    constexpr int MAXD = 256;
    __shared__ __align__(16) __half sm[2][TILE_TOK][MAXD + 8];
    const int j = blockIdx.x, g = blockIdx.y;
    const int t0 = j * TILE_TOK;
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
    const int64_t piece = 2 * D;                              // uint4 per tile piece (32 * D bytes)
    uint4* kout = out + ((int64_t)g * 2 * ntiles + j) * piece;
    uint4* vout = out + ((int64_t)g * 2 * ntiles + ntiles + j) * piece;
    const int cpt = D / 8;                                    // d chunks (K) / d groups (V)
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
    if (src_f16)
        quantize_mlx4g32_kernel<__half><<<blocks, threads, 0, st>>>(static_cast<const __half*>(X), rows, kv_dim,
                                                                     static_cast<uint8_t*>(out));
    else
        quantize_mlx4g32_kernel<float><<<blocks, threads, 0, st>>>(static_cast<const float*>(X), rows, kv_dim,
                                                                    static_cast<uint8_t*>(out));
    return cudaGetLastError();
}

cudaError_t launch_relayout_fp16(const void* K, const void* V, int src_f16, int H_kv, int N, int D, int ntiles,
                                 void* out, cudaStream_t st, int sms) {
    (void)sms;
    if (D > 256 || D % 8 != 0) return cudaErrorInvalidValue;
    const dim3 grid(ntiles, H_kv);
    if (src_f16)
        relayout_fp16_kernel<__half><<<grid, 128, 0, st>>>(static_cast<const __half*>(K), static_cast<const __half*>(V),
                                                           N, D, ntiles, static_cast<uint4*>(out));
    else
        relayout_fp16_kernel<float><<<grid, 128, 0, st>>>(static_cast<const float*>(K), static_cast<const float*>(V),
                                                          N, D, ntiles, static_cast<uint4*>(out));
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
