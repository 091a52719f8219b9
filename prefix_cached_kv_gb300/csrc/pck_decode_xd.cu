// pck_decode_xd.cu -- the split-K decode (pck_decode_impl.cuh) for the head dimensions 32, 96,
// 160, 192 and 512 that the pages' kernels also serve ("ATTEND.* and ATTEND.PREFIX.*": one pipeline
// per D in {32, 64, 96, 128, 160, 192, 256, 512}). fp16 slots take all five (D = 512 with q in
// shared memory, one ring stage per warp and at most 4 q heads per work group); the mlx4g32
// fragment layout packs 64 dimensions per 16-byte load, so mlx4g32 slots take 192 here (and 64,
// 128, 256 in pck_decode.cu).
#include "pck_decode_impl.cuh"

namespace pck {

bool decode_dim_ok(int fmt, int D) {
    if (D == 64 || D == 128 || D == 256 || D == 192) return true;
    return fmt == FMT_FP16 && (D == 32 || D == 96 || D == 160 || D == 512);
}

DecodeLaunchInfo decode_launch_info_xd(int fmt, int D, int ncb) {
    if (fmt == FMT_FP16) {
        if (D == 32) return info_d<FMT_FP16, 32>(ncb);
        if (D == 96) return info_d<FMT_FP16, 96>(ncb);
        if (D == 160) return info_d<FMT_FP16, 160>(ncb);
        if (D == 192) return info_d<FMT_FP16, 192>(ncb);
        if (D == 512) return info_d<FMT_FP16, 512>(ncb);
    } else if (D == 192) {
        return info_d<FMT_I4, 192>(ncb);
    }
    return DecodeLaunchInfo{0, 0, 0, 1};
}

cudaError_t launch_decode_xd(int fmt, int D, const DecodeParams& p, int n_ctas, cudaStream_t st) {
    const int ncb = decode_ncb(p);
    if (fmt == FMT_FP16) {
        if (D == 32) return launch_d<FMT_FP16, 32>(p, ncb, n_ctas, st);
        if (D == 96) return launch_d<FMT_FP16, 96>(p, ncb, n_ctas, st);
        if (D == 160) return launch_d<FMT_FP16, 160>(p, ncb, n_ctas, st);
        if (D == 192) return launch_d<FMT_FP16, 192>(p, ncb, n_ctas, st);
        if (D == 512) return launch_d<FMT_FP16, 512>(p, ncb, n_ctas, st);
    } else if (D == 192) {
        return launch_d<FMT_I4, 192>(p, ncb, n_ctas, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace pck
