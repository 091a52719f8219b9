// pck_select.cuh -- warp-level top-K helpers shared by the block-mean selectors (the selection
// kernel of pck_sparse.cu and the fused sparse kernel of pck_sparse_fused.cu).
#pragma once

#include <stdint.h>

namespace pck {

// Selection order: higher score first, ties to the lower block index. A score and its block
// become one 64-bit key whose unsigned order is that order (the float's bits made monotone,
// then the block index inverted), so every comparison below is a branch-free integer compare.
// Key 0 stands for "no block".
__device__ __forceinline__ uint64_t score_key(float s, int b) {
    const uint32_t u = __float_as_uint(s == 0.f ? 0.f : s);   // -0 ties with +0
    const uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return (static_cast<uint64_t>(o) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(b));
}
__device__ __forceinline__ int key_block(uint64_t k) { return static_cast<int>(~static_cast<uint32_t>(k)); }
__device__ __forceinline__ uint64_t umax64(uint64_t a, uint64_t b) { return a > b ? a : b; }
__device__ __forceinline__ uint64_t shfl64(uint64_t v, int src) {
    const uint32_t lo = __shfl_sync(0xffffffffu, static_cast<uint32_t>(v), src);
    const uint32_t hi = __shfl_sync(0xffffffffu, static_cast<uint32_t>(v >> 32), src);
    return (static_cast<uint64_t>(hi) << 32) | lo;
}
__device__ __forceinline__ uint64_t shfl64_xor(uint64_t v, int m) {
    const uint32_t lo = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(v), m);
    const uint32_t hi = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(v >> 32), m);
    return (static_cast<uint64_t>(hi) << 32) | lo;
}
__device__ __forceinline__ uint64_t max32(const uint64_t (&k)[32]) {   // a depth-5 tree
    uint64_t t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) t[i] = umax64(k[2 * i], k[2 * i + 1]);
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) t[i] = umax64(t[2 * i], t[2 * i + 1]);
    return t[0];
}

// Top-K of one q head's keys held 32 per lane, when K <= 32: every lane takes its best key;
// the K-th best of those 32 lane bests, T, bounds the answer (the K lane bests ranked 0..K-1
// are all >= T, so the K-th best key is too), so the top K are among the keys >= T. When
// there are at most 32 of them they are gathered and each one's rank among them is its place;
// otherwise (many ties) the caller falls back to K rounds of arg-max. picks[r] = r-th best.
__device__ __forceinline__ bool topk_by_threshold(const uint64_t (&key)[32], int K, int lane, uint64_t* cand,
                                                  int* picks) {
    const uint64_t m = max32(key);
    int rank = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) rank += shfl64(m, j) > m ? 1 : 0;
    const unsigned at = __ballot_sync(0xffffffffu, m != 0 && rank == K - 1);
    if (at == 0u) return false;
    const uint64_t T = shfl64(m, __ffs(at) - 1);
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) cnt += key[i] >= T ? 1 : 0;
    int pre = cnt;   // inclusive scan over lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, pre, o);
        pre += lane >= o ? x : 0;
    }
    const int C = __shfl_sync(0xffffffffu, pre, 31);
    if (C > 32) return false;
    int pos = pre - cnt;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        if (key[i] >= T) cand[pos] = key[i];
        pos += key[i] >= T ? 1 : 0;
    }
    __syncwarp();
    if (lane < C) {
        const uint64_t k = cand[lane];
        int r = 0;
        for (int j = 0; j < C; ++j) r += cand[j] > k ? 1 : 0;
        if (r < K) picks[r] = key_block(k);
    }
    __syncwarp();
    return true;
}

}  // namespace pck
