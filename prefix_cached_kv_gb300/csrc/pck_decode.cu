// pck_decode.cu -- the split-K decode (pck_decode_impl.cuh) for head dimensions 64, 128 and 256,
// the launch planning, and the dispatch of a launch to its instantiation.
#include <algorithm>

#include "pck_decode_impl.cuh"

namespace pck {

// ncb: 4-head column blocks of the mlx4g32 kernel (1 when every work group has <= 4 q heads).
DecodeLaunchInfo decode_launch_info(int fmt, int D, int ncb) {
    if (fmt == FMT_FP16) {
        if (D == 64) return info_d<FMT_FP16, 64>(ncb);
        if (D == 128) return info_d<FMT_FP16, 128>(ncb);
        if (D == 256) return info_d<FMT_FP16, 256>(ncb);
    } else {
        if (D == 64) return info_d<FMT_I4, 64>(ncb);
        if (D == 128) return info_d<FMT_I4, 128>(ncb);
        if (D == 256) return info_d<FMT_I4, 256>(ncb);
    }
    return decode_launch_info_xd(fmt, D, ncb);
}

bool plan_decode(DecodeParams* p, int64_t total, int vmax, int n_items, int S_suf, int sms, int ctas_per_sm,
                 int64_t max_slots, DecodePlan* out) {
    const bool sparse = p->sparse != 0;
    const int n_suf = (S_suf + TILE_TOK - 1) / TILE_TOK;
    const int64_t n_suf_warps = static_cast<int64_t>(n_items) * n_suf;
    const int64_t fixed = n_items + n_suf_warps;            // item slots + suffix piece slots
    if (fixed >= max_slots) return false;
    // prefix workers and suffix warps together stay within one wave of resident warps
    int64_t max_warps = static_cast<int64_t>(sms) * ctas_per_sm * DECODE_WARPS - n_suf_warps;
    if (max_warps < 1) max_warps = 1;
    if (max_warps > max_slots - fixed) max_warps = max_slots - fixed;
    int64_t tpw = (total + max_warps - 1) / max_warps;
    tpw = std::max<int64_t>(tpw, std::max<int64_t>((vmax + 63) / 64, 4));   // at most ~64 pieces per item, at least 4 tiles each
    if (tpw < 2) tpw = 2;
    int64_t n_workers = 0;
    p->aligned = 0;
    if (sparse) {
        n_workers = std::min<int64_t>(max_warps, total);
    } else {
        // whole pieces per item; grow the target size until the pieces fit the warps
        const int64_t tpw0 = tpw;
        for (;; ++tpw) {
            n_workers = 0;
            for (int d = 0; d < p->n_desc; ++d) {
                const int vt = p->desc[d].vtiles;
                const int ps = static_cast<int>(std::min<int64_t>(vt, (vt + ((vt + tpw - 1) / tpw) - 1) / ((vt + tpw - 1) / tpw)));
                p->ppi[d] = (vt + ps - 1) / ps;                  // every piece non-empty
                p->wbase[d] = static_cast<int>(n_workers);
                n_workers += static_cast<int64_t>(p->n_groups) * p->ppi[d];
            }
            p->wbase[p->n_desc] = static_cast<int>(n_workers);
            if (n_workers <= max_warps || tpw >= vmax) break;
        }
        int max_ps = 1;
        for (int d = 0; d < p->n_desc; ++d)
            max_ps = std::max(max_ps, (p->desc[d].vtiles + p->ppi[d] - 1) / p->ppi[d]);
        if (n_workers <= max_warps && max_ps * 20 <= tpw0 * 21) {
            p->aligned = 1;
        } else {   // plain ranges of tpw0 tiles across the items
            tpw = tpw0;
            n_workers = (total + tpw - 1) / tpw;
        }
        if (n_workers + fixed > max_slots) return false;
    }
    out->tpw = static_cast<int>(tpw);
    out->n_workers = static_cast<int>(n_workers);
    out->n_suf = n_suf;
    out->n_ctas = static_cast<int>((n_workers + n_suf_warps + DECODE_WARPS - 1) / DECODE_WARPS);
    out->slots = n_workers + fixed;
    return true;
}

int decode_ncb(const DecodeParams& p) {
    int mx = 0;
    for (int i = 0; i < p.n_groups; ++i) mx = p.grp[i].nq > mx ? p.grp[i].nq : mx;
    return mx > 4 ? 2 : 1;
}

cudaError_t launch_decode(int fmt, int D, const DecodeParams& p, int n_ctas, cudaStream_t st) {
    const int ncb = decode_ncb(p);
    if (fmt == FMT_FP16) {
        if (D == 64) return launch_d<FMT_FP16, 64>(p, ncb, n_ctas, st);
        if (D == 128) return launch_d<FMT_FP16, 128>(p, ncb, n_ctas, st);
        if (D == 256) return launch_d<FMT_FP16, 256>(p, ncb, n_ctas, st);
    } else {
        if (D == 64) return launch_d<FMT_I4, 64>(p, ncb, n_ctas, st);
        if (D == 128) return launch_d<FMT_I4, 128>(p, ncb, n_ctas, st);
        if (D == 256) return launch_d<FMT_I4, 256>(p, ncb, n_ctas, st);
    }
    return launch_decode_xd(fmt, D, p, n_ctas, st);
}

}  // namespace pck
