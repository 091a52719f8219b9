// pck_noalloc.cu -- M=1 attention over caller-held mlx4g32 records that allocates nothing.
//
// Some callers cannot allocate device memory when they need an answer: code that runs inside
// another framework's memory budget (its caching allocator owns the device heap), a serving
// loop that is forbidden to touch the allocator on the request path, or a process that has
// not created a pck context at all. For them, pck_attend_records_noalloc runs the same two
// kernels as a store + fused query (records -> resident tiles, then the split-K decode with
// the suffix merge), planned by the same split as the context path, but every scratch byte it
// needs lives in the file-scope device arrays below instead of memory from cudaMalloc. The
// caller passes only inputs and outputs.
//
// Cost of that choice: every GPU that loads libpck holds these arrays (PCK_NOALLOC_SCRATCH_BYTES
// in total) until the process exits, and all calls share them, so calls that overlap on the
// GPU (two streams, or two host threads) race and must be serialised by the caller.
//
// The kernels' device error codes (a bounded wait that gave up, a Q element out of range) land
// in the scratch's error word, which keeps them until pck_noalloc_status reads and clears it.
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/pck.h"
#include "pck_common.cuh"
#include "pck_kernels.h"

namespace {

using namespace pck;

constexpr size_t NA_TILE_BYTES = size_t(16) << 20;      // resident tiles of one query's slot
constexpr size_t NA_PARTIAL_BYTES = size_t(16) << 20;   // split-K partials
constexpr int NA_MAX_DEVICES = 64;

static __device__ __align__(256) uint8_t g_na_tiles[NA_TILE_BYTES];
static __device__ __align__(256) float g_na_partials[NA_PARTIAL_BYTES / sizeof(float)];
static __device__ __align__(256) int g_na_err[64];

static_assert(NA_TILE_BYTES + NA_PARTIAL_BYTES + 64 * sizeof(int) == PCK_NOALLOC_SCRATCH_BYTES,
              "the header states the scratch size");

// Per device: the scratch arrays' device addresses (host code must not pass the symbols
// themselves: in host code they are host-side stand-ins), the SM count and the decode
// kernels' occupancy, found once with the device current.
struct NaDevice {
    std::once_flag once;
    int rc = PCK_ECUDA;
    uint8_t* tiles = nullptr;
    float* partials = nullptr;
    int* err = nullptr;
    int sms = 0;
    int ctas_per_sm[4][2] = {};   // [D = 64, 128, 192, 256][column blocks 1, 2]
};
NaDevice g_na[NA_MAX_DEVICES];

void na_setup_once(NaDevice& s, int dev) {
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&s.tiles), g_na_tiles) != cudaSuccess ||
        cudaGetSymbolAddress(reinterpret_cast<void**>(&s.partials), g_na_partials) != cudaSuccess ||
        cudaGetSymbolAddress(reinterpret_cast<void**>(&s.err), g_na_err) != cudaSuccess ||
        cudaDeviceGetAttribute(&s.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || s.sms <= 0) {
        cudaGetLastError();
        s.rc = PCK_ECUDA;
        return;
    }
    const int Ds[4] = {64, 128, 192, 256};
    for (int i = 0; i < 4; ++i)
        for (int ncb = 1; ncb <= 2; ++ncb) s.ctas_per_sm[i][ncb - 1] = decode_launch_info(FMT_I4, Ds[i], ncb).ctas_per_sm;
    s.rc = cudaGetLastError() == cudaSuccess ? PCK_OK : PCK_ECUDA;
}

// The current device's scratch, set up on first use (thread-safe: one set-up per device).
NaDevice* na_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= NA_MAX_DEVICES) return nullptr;
    NaDevice& s = g_na[dev];
    std::call_once(s.once, [&s, dev] { na_setup_once(s, dev); });
    return s.rc == PCK_OK ? &s : nullptr;
}

}  // namespace

extern "C" int pck_attend_records_noalloc(int H_kv, int N, int D, const void* K_rec, const void* V_rec, int H_q,
                                          int q_dtype, const void* Q, const int32_t* head_map, int S_suf,
                                          const void* K_suf, const void* V_suf, float* O, float* LSE,
                                          void* stream) {
    using namespace pck;
    if (!K_rec || !V_rec || !Q || !O) return PCK_EINVAL;
    if ((reinterpret_cast<uintptr_t>(O) | reinterpret_cast<uintptr_t>(Q)) & 15) return PCK_EINVAL;
    if (H_kv < 1 || H_kv > PCK_MAX_HEADS || H_q < 1 || H_q > PCK_MAX_HEADS || N < 1 || S_suf < 0) return PCK_EINVAL;
    if (D != 64 && D != 128 && D != 192 && D != 256) return PCK_EUNSUPPORTED;
    if (q_dtype != PCK_DT_F32 && q_dtype != PCK_DT_F16) return PCK_EINVAL;
    if (S_suf > 0 && (!K_suf || !V_suf)) return PCK_EINVAL;
    if ((reinterpret_cast<uintptr_t>(K_rec) | reinterpret_cast<uintptr_t>(V_rec)) & 3) return PCK_EINVAL;

    // q heads grouped by kv head, at most GMAX per group (host-only work before any CUDA call)
    int hm[PCK_MAX_HEADS];
    for (int h = 0; h < H_q; ++h) {
        if (head_map) {
            hm[h] = head_map[h];
        } else {
            if (H_q % H_kv) return PCK_EINVAL;
            hm[h] = h / (H_q / H_kv);
        }
        if (hm[h] < 0 || hm[h] >= H_kv) return PCK_EINVAL;
    }
    static thread_local DecodeParams p;
    std::memset(&p, 0, sizeof p);
    int n_groups = 0, max_nq = 0;
    for (int g = 0; g < H_kv; ++g) {
        WorkGroup cur{g, 0, {-1, -1, -1, -1, -1, -1, -1, -1}};
        for (int h = 0; h < H_q; ++h) {
            if (hm[h] != g) continue;
            cur.qh[cur.nq++] = static_cast<int8_t>(h);
            if (cur.nq == GMAX) {
                p.grp[n_groups++] = cur;
                cur = WorkGroup{g, 0, {-1, -1, -1, -1, -1, -1, -1, -1}};
            }
        }
        if (cur.nq) p.grp[n_groups++] = cur;
    }
    for (int i = 0; i < n_groups; ++i) max_nq = p.grp[i].nq > max_nq ? p.grp[i].nq : max_nq;

    // size limit of the static tile scratch
    const int ntiles = (N + TILE_TOK - 1) / TILE_TOK;
    const size_t tiles_bytes = static_cast<size_t>(H_kv) * ntiles * tile_bytes(FMT_I4, D);
    if (tiles_bytes > NA_TILE_BYTES) return PCK_EUNSUPPORTED;

    NaDevice* sp = na_device();
    if (!sp) return PCK_ECUDA;
    const int ncb = max_nq > 4 ? 2 : 1;
    const int di = D == 64 ? 0 : (D == 128 ? 1 : (D == 192 ? 2 : 3));
    const int64_t total = static_cast<int64_t>(n_groups) * ntiles;
    const int64_t max_slots =
        static_cast<int64_t>(NA_PARTIAL_BYTES / (static_cast<size_t>(GMAX) * partial_stride(D) * sizeof(float)));
    DecodePlan plan;
    p.n_desc = 1;
    p.n_groups = n_groups;
    p.desc[0].vtiles = ntiles;
    if (!plan_decode(&p, total, ntiles, n_groups, S_suf, sp->sms, sp->ctas_per_sm[di][ncb - 1], max_slots, &plan))
        return PCK_EUNSUPPORTED;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (launch_relayout_mlx4(K_rec, V_rec, 0, H_kv, N, D, ntiles, sp->tiles, st, sp->sms) != cudaSuccess)
        return PCK_ECUDA;

    p.n_desc = 1;
    p.n_groups = n_groups;
    p.H_q = H_q;
    p.H_kv = H_kv;
    p.S_suf = S_suf;
    p.q_f16 = q_dtype == PCK_DT_F16;
    p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
    DecodeDesc& d = p.desc[0];
    d.kv = sp->tiles;
    d.Q = Q;
    d.O = O;
    d.LSE = LSE;
    d.Ksuf = static_cast<const __half*>(K_suf);
    d.Vsuf = static_cast<const __half*>(V_suf);
    d.N = N;
    d.ntiles = ntiles;
    d.vtiles = ntiles;
    d.tile_off = 0;
    p.total_tiles = static_cast<int>(total);
    p.tpw = plan.tpw;
    p.max_units = static_cast<int>(total);
    p.n_workers = plan.n_workers;
    p.n_suf = plan.n_suf;
    p.partials = sp->partials;
    p.counters = nullptr;   // the dense decode takes no tickets
    p.err = sp->err;
    if (launch_decode(FMT_I4, D, p, plan.n_ctas, st) != cudaSuccess) return PCK_ECUDA;
    return PCK_OK;
}

extern "C" int pck_noalloc_status(void* stream, int* code) {
    using namespace pck;
    if (code) *code = 0;
    NaDevice* sp = na_device();
    if (!sp) return PCK_ECUDA;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return PCK_ECUDA;
    }
    int h = 0;
    if (cudaMemcpy(&h, sp->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return PCK_ECUDA;
    }
    if (code) *code = h;
    if (h == 0) return PCK_OK;
    if (cudaMemset(sp->err, 0, sizeof(int)) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
    }
    return PCK_ECUDA;
}
