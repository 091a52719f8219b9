// pck_api.cu -- host runtime and C ABI of libpck (declared in include/pck.h).
//
// Slot table: resident (sid, layer) entries, the problem statement of ATTEND.PREFIX.STORE /
// LOOKUP ("ATTEND.* and ATTEND.PREFIX.*", section "Wire forms"). When the table is full the
// least recently used slot is released and its key kept in a bounded cold registry, so that a
// later query answers PCK_COLDMISS instead of PCK_MISS ("Shared KV Cache Serving -- Pion as LLM
// Memory", section "Cold-tier state machine": WARM / COLD / MISSING).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <deque>
#include <list>
#include <string>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "../../include/pck.h"
#include "pck_common.cuh"
#include "pck_kernels.h"

using namespace pck;

namespace {

constexpr int COLD_SLOTS = 1024;
constexpr size_t WS_PARTIAL_BYTES = size_t(64) << 20;  // split-K partials
constexpr int WS_COUNTERS = 1 << 16;
constexpr int WS_SEL_BYTES = 1 << 20;                   // sparse selection lists
constexpr size_t WS_SCORES_BYTES = size_t(16) << 20;
constexpr size_t WS_SUFFIX_BYTES = size_t(32) << 20;    // batched-Q suffix staged in the slot layout
constexpr size_t ARENA_CHUNK = size_t(256) << 20;      // block-means arena: chunk size
constexpr size_t ARENA_ALIGN = 256;

// The block means of every slot (fp32 and split), packed side by side into a few large chunks
// instead of one pool allocation each between the slots' tiles: the batched sparse kernel
// streams the means of many sessions at once, and packed together they read ~11 % faster
// (0.65 against 0.73 us per session on the 64-session sparse batch). A freed range is reused
// once the work its freeing stream had queued has completed (an event recorded there).
struct MeansArena {
    struct Chunk {
        uint8_t* base;
        size_t size, top;
    };
    struct Range {
        uint8_t* p;
        size_t bytes;
        cudaEvent_t ready;   // nullptr: reusable now
    };
    std::vector<Chunk> chunks;
    std::vector<Range> freed;
};

struct Slot {
    int fmt = 0, H_kv = 0, N = 0, D = 0, ntiles = 0;
    uint8_t* tiles = nullptr;
    size_t bytes = 0;
    std::unordered_map<int, float*> kmean;  // block size -> [H_kv, nb, D] fp32 (in the means arena)
    // block size -> the same means as fp16 hi + lo pairs in the tensor-core tile layout (16 blocks
    // a tile, [H_kv][ceil(nb / 16)][hi part | lo part]; see launch_block_means_split)
    std::unordered_map<int, uint8_t*> kmean_split;
    std::list<std::string>::iterator lru;
};

}  // namespace

struct pck_ctx {
    int device = 0;
    int sms = 0;
    int max_slots = 256;
    std::string err;
    std::unordered_map<std::string, Slot> slots;
    std::list<std::string> lru;                 // front = most recent
    std::deque<std::string> cold_fifo;
    std::unordered_set<std::string> cold;
    float* partials = nullptr;
    int* counters = nullptr;
    int* dev_err = nullptr;
    uint8_t* sel = nullptr;
    float* scores = nullptr;
    uint8_t* suf_ws = nullptr;
    uint8_t* host_stage = nullptr;   // host-buffer calls: their inputs, copied in (PCK_HOST_STAGE_BYTES)
    MeansArena means;
    int64_t queries = 0, stores = 0, evictions = 0;
    int64_t bytes_resident = 0;
    DecodeLaunchInfo dinfo[2][16];   // [format][head dimension x column blocks]
    bool dinfo_ok[2][16] = {};
};

namespace {

int fail(pck_ctx* c, int code, const char* fmt, ...) {
    if (c) {
        char buf[512];
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(buf, sizeof buf, fmt, ap);
        va_end(ap);
        c->err = buf;
    }
    return code;
}

int cuda_fail(pck_ctx* c, cudaError_t e, const char* what) {
    return fail(c, PCK_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

std::string key_of(const char* sid, int layer) {
    std::string k(sid);
    k.push_back('\x1f');
    k += std::to_string(layer);
    return k;
}

// head dimensions with kernels, per resident format (the M=1 kernels; M>1 and the sparse forms
// check their own)
bool d_ok(int D, int fmt) { return decode_dim_ok(fmt == PCK_FMT_FP16 ? FMT_FP16 : FMT_I4, D); }
int d_index(int D) {
    switch (D) {
        case 32: return 0;
        case 64: return 1;
        case 96: return 2;
        case 128: return 3;
        case 160: return 4;
        case 192: return 5;
        case 256: return 6;
        default: return 7;
    }
}

// q heads per work group: D = 512 keeps one column block of 4 heads (its O accumulators fill a
// lane's registers), so a kv head with more q heads is read once per 4 of them.
int d_gmax(int D) { return D >= 512 ? 4 : GMAX; }

const DecodeLaunchInfo& dinfo(pck_ctx* c, int fmt, int D, int ncb) {
    const int i = d_index(D) + 8 * (ncb - 1);
    if (!c->dinfo_ok[fmt][i]) {
        c->dinfo[fmt][i] = decode_launch_info(fmt, D, ncb);
        c->dinfo_ok[fmt][i] = true;
    }
    return c->dinfo[fmt][i];
}

bool capturing(cudaStream_t st) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
        cudaGetLastError();
        return true;
    }
    return cs != cudaStreamCaptureStatusNone;
}

size_t arena_round(size_t bytes) { return (bytes + ARENA_ALIGN - 1) & ~(ARENA_ALIGN - 1); }

// A range of the means arena: a freed range whose stream work has completed, else the top of a
// chunk, else a new chunk (nullptr when the device is out of memory).
uint8_t* arena_alloc(pck_ctx* c, size_t bytes) {
    bytes = arena_round(bytes);
    MeansArena& A = c->means;
    for (size_t i = 0; i < A.freed.size(); ++i) {
        MeansArena::Range& r = A.freed[i];
        if (r.bytes < bytes) continue;
        if (r.ready) {
            if (cudaEventQuery(r.ready) != cudaSuccess) {
                cudaGetLastError();   // not ready yet (or a sticky error, reported by the next call)
                continue;
            }
            cudaEventDestroy(r.ready);
            r.ready = nullptr;
        }
        uint8_t* p = r.p;
        if (r.bytes == bytes) {
            A.freed.erase(A.freed.begin() + static_cast<std::ptrdiff_t>(i));
        } else {
            r.p += bytes;
            r.bytes -= bytes;
        }
        return p;
    }
    for (MeansArena::Chunk& ch : A.chunks)
        if (ch.size - ch.top >= bytes) {
            uint8_t* p = ch.base + ch.top;
            ch.top += bytes;
            return p;
        }
    const size_t sz = std::max(ARENA_CHUNK, bytes);
    uint8_t* base = nullptr;
    if (cudaMalloc(reinterpret_cast<void**>(&base), sz) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    A.chunks.push_back({base, sz, bytes});
    return base;
}

// Returns a range to the arena once the work queued on st so far (the last reads of it in stream
// order) has completed. Without an event the range stays unused until the context ends.
void arena_free(pck_ctx* c, void* p, size_t bytes, cudaStream_t st) {
    cudaEvent_t ev = nullptr;
    if (capturing(st) || cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventRecord(ev, st) != cudaSuccess) {
        cudaGetLastError();
        if (ev) cudaEventDestroy(ev);
        return;
    }
    c->means.freed.push_back({static_cast<uint8_t*>(p), arena_round(bytes), ev});
}

size_t kmean_bytes(const Slot& s, int B) { return static_cast<size_t>(s.H_kv) * ((s.N + B - 1) / B) * s.D * sizeof(float); }
size_t kmean_split_bytes(const Slot& s, int B) {
    return static_cast<size_t>(s.H_kv) * (((s.N + B - 1) / B + 15) / 16) * 64 * s.D;
}

void free_slot(pck_ctx* c, Slot& s, cudaStream_t st) {
    if (s.tiles) cudaFreeAsync(s.tiles, st);
    for (auto& kv : s.kmean) arena_free(c, kv.second, kmean_bytes(s, kv.first), st);
    for (auto& kv : s.kmean_split) arena_free(c, kv.second, kmean_split_bytes(s, kv.first), st);
    c->bytes_resident -= static_cast<int64_t>(s.bytes);
    s.tiles = nullptr;
    s.kmean.clear();
    s.kmean_split.clear();
}

void remember_cold(pck_ctx* c, const std::string& k) {
    if (c->cold.count(k)) return;
    c->cold.insert(k);
    c->cold_fifo.push_back(k);
    if (static_cast<int>(c->cold_fifo.size()) > COLD_SLOTS) {
        c->cold.erase(c->cold_fifo.front());
        c->cold_fifo.pop_front();
    }
}

void forget_cold(pck_ctx* c, const std::string& k) {
    if (!c->cold.erase(k)) return;
    for (auto it = c->cold_fifo.begin(); it != c->cold_fifo.end(); ++it)
        if (*it == k) { c->cold_fifo.erase(it); break; }
}

// Look up a resident slot and mark it most recently used; status PCK_OK / PCK_MISS / PCK_COLDMISS.
int find_slot(pck_ctx* c, const char* sid, int layer, Slot** out) {
    if (!sid) return fail(c, PCK_EINVAL, "sid is NULL");
    const std::string k = key_of(sid, layer);
    auto it = c->slots.find(k);
    if (it == c->slots.end()) {
        if (c->cold.count(k)) return fail(c, PCK_COLDMISS, "COLDMISS %s layer %d (evicted)", sid, layer);
        return fail(c, PCK_MISS, "session not found: %s layer %d", sid, layer);
    }
    c->lru.splice(c->lru.begin(), c->lru, it->second.lru);
    *out = &it->second;
    return PCK_OK;
}

// Insert (replacing any previous slot with the key), evicting the LRU slot when full.
Slot* put_slot(pck_ctx* c, const std::string& k, cudaStream_t st) {
    auto it = c->slots.find(k);
    if (it != c->slots.end()) {
        free_slot(c, it->second, st);
        c->lru.erase(it->second.lru);
        c->slots.erase(it);
    }
    while (static_cast<int>(c->slots.size()) >= c->max_slots && !c->lru.empty()) {
        const std::string victim = c->lru.back();
        auto v = c->slots.find(victim);
        free_slot(c, v->second, st);
        c->slots.erase(v);
        c->lru.pop_back();
        remember_cold(c, victim);
        ++c->evictions;
    }
    forget_cold(c, k);
    c->lru.push_front(k);
    Slot& s = c->slots[k];
    s.lru = c->lru.begin();
    return &s;
}

int check_async(pck_ctx* c) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(c, e, "CUDA error");
    return PCK_OK;
}

// q heads grouped by kv head, at most gmax (<= GMAX) per work group.
int build_groups(pck_ctx* c, int H_q, int H_kv, const int32_t* head_map, WorkGroup* grp, int* n_groups,
                 int8_t* hm_out, int* max_nq, int gmax = GMAX) {
    if (H_q < 1 || H_kv < 1 || H_q > PCK_MAX_HEADS || H_kv > PCK_MAX_HEADS)
        return fail(c, PCK_EINVAL, "H_q=%d H_kv=%d out of range [1, %d]", H_q, H_kv, PCK_MAX_HEADS);
    int hm[PCK_MAX_HEADS];
    for (int h = 0; h < H_q; ++h) {
        if (head_map) {
            hm[h] = head_map[h];
        } else {
            if (H_q % H_kv) return fail(c, PCK_EINVAL, "H_q=%d not a multiple of H_kv=%d and no head_map", H_q, H_kv);
            hm[h] = h / (H_q / H_kv);
        }
        if (hm[h] < 0 || hm[h] >= H_kv) return fail(c, PCK_EINVAL, "head_map[%d]=%d outside [0, %d)", h, hm[h], H_kv);
        if (hm_out) hm_out[h] = static_cast<int8_t>(hm[h]);
    }
    int n = 0, mx = 0;
    for (int g = 0; g < H_kv; ++g) {
        WorkGroup cur{g, 0, {-1, -1, -1, -1, -1, -1, -1, -1}};
        for (int h = 0; h < H_q; ++h) {
            if (hm[h] != g) continue;
            cur.qh[cur.nq++] = static_cast<int8_t>(h);
            if (cur.nq == gmax) {
                if (n == MAX_GROUPS) return fail(c, PCK_EUNSUPPORTED, "too many work groups");
                grp[n++] = cur;
                mx = gmax;
                cur = WorkGroup{g, 0, {-1, -1, -1, -1, -1, -1, -1, -1}};
            }
        }
        if (cur.nq) {
            if (n == MAX_GROUPS) return fail(c, PCK_EUNSUPPORTED, "too many work groups");
            mx = std::max(mx, cur.nq);
            grp[n++] = cur;
        }
    }
    *n_groups = n;
    if (max_nq) *max_nq = mx;
    return PCK_OK;
}

struct DescIn {
    Slot* slot;
    const void* Q;
    float* O;
    float* LSE;
    const void* Ksuf;
    const void* Vsuf;
    const int* sel_blocks = nullptr;     // sparse: the query's [n_groups, sel_max] block lists
    const uint8_t* sel_mask = nullptr;   // sparse: per-block q-head masks
    int window = 0;                      // dense M=1: fa_window (0: none)
};

// Plan and launch one decode over n descriptors (dense), or one sparse descriptor.
int run_decode(pck_ctx* c, int fmt, int D, int H_q, int H_kv, int S_suf, int q_f16, const WorkGroup* grp,
               int n_groups, const DescIn* dsc, int n, int sparse, int tiles_per_block, int sel_max, const int* item_base,
               cudaStream_t st) {
    static thread_local DecodeParams p;   // ~6 KB, built on the host and copied into the launch
    std::memset(&p, 0, sizeof p);
    p.n_desc = n;
    p.n_groups = n_groups;
    p.H_q = H_q;
    p.H_kv = H_kv;
    p.S_suf = S_suf;
    p.q_f16 = q_f16;
    p.sparse = sparse;
    p.tiles_per_block = tiles_per_block;
    p.sel_max = sel_max;
    p.item_base = item_base;
    p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
    for (int g = 0; g < n_groups; ++g) p.grp[g] = grp[g];
    int64_t total = 0;
    for (int i = 0; i < n; ++i) {
        DecodeDesc& d = p.desc[i];
        d.kv = dsc[i].slot->tiles;
        d.Q = dsc[i].Q;
        d.O = dsc[i].O;
        d.LSE = dsc[i].LSE;
        d.Ksuf = static_cast<const __half*>(dsc[i].Ksuf);
        d.Vsuf = static_cast<const __half*>(dsc[i].Vsuf);
        d.N = dsc[i].slot->N;
        d.ntiles = dsc[i].slot->ntiles;
        d.t_lo = d.s_lo = d.tile0 = 0;
        if (!sparse && dsc[i].window > 0) {   // the last `window` positions of prefix + suffix
            const int first = d.N + S_suf - dsc[i].window;   // first visible position
            d.t_lo = std::min(std::max(first, 0), d.N);      // == N: no prefix token is visible
            d.s_lo = std::max(first - d.N, 0);
            d.tile0 = std::min(d.t_lo, d.N - 1) / TILE_TOK;  // keep one (masked) tile
        }
        d.vtiles = sparse ? sel_max * tiles_per_block : d.ntiles - d.tile0;
        d.sel_blocks = dsc[i].sel_blocks;
        d.sel_mask = dsc[i].sel_mask;
        d.tile_off = static_cast<int>(total);
        total += static_cast<int64_t>(n_groups) * d.vtiles;
    }
    if (total >= (int64_t(1) << 30)) return fail(c, PCK_EUNSUPPORTED, "too many tiles in one launch");
    const DecodeLaunchInfo& li = dinfo(c, fmt, D, decode_ncb(p));
    int vmax = 1;
    for (int i = 0; i < n; ++i) vmax = std::max(vmax, p.desc[i].vtiles);
    const int n_items = n * n_groups;
    if (n_items > WS_COUNTERS) return fail(c, PCK_EUNSUPPORTED, "too many work items");
    const int64_t max_slots =
        static_cast<int64_t>(WS_PARTIAL_BYTES / (static_cast<size_t>(GMAX) * partial_stride(D) * sizeof(float)));
    DecodePlan plan;
    if (!plan_decode(&p, total, vmax, n_items, S_suf, c->sms, li.ctas_per_sm, max_slots, &plan))
        return fail(c, PCK_EUNSUPPORTED, "split-K workspace too small for %d items", n_items);
    p.total_tiles = static_cast<int>(total);
    p.tpw = plan.tpw;
    p.max_units = static_cast<int>(total);
    p.n_workers = plan.n_workers;
    p.n_suf = plan.n_suf;
    p.partials = c->partials;
    p.counters = c->counters;
    p.err = c->dev_err;
    const int n_ctas = plan.n_ctas;
    cudaError_t e = launch_decode(fmt, D, p, n_ctas, st);
    if (e != cudaSuccess) return cuda_fail(c, e, "decode launch");
    ++c->queries;
    return PCK_OK;
}

bool dtype_ok(int dt) { return dt == PCK_DT_F32 || dt == PCK_DT_F16; }

}  // namespace

extern "C" {

int pck_create(pck_ctx** out, int device, int max_slots) {
    if (!out) return PCK_EINVAL;
    *out = nullptr;
    cudaError_t e = cudaSetDevice(device);
    if (e != cudaSuccess) return PCK_ECUDA;
    pck_ctx* c = new pck_ctx();
    c->device = device;
    c->max_slots = max_slots > 0 ? max_slots : 256;
    cudaDeviceGetAttribute(&c->sms, cudaDevAttrMultiProcessorCount, device);
    if (c->sms <= 0) c->sms = 1;
    if (cudaMalloc(&c->partials, WS_PARTIAL_BYTES) != cudaSuccess ||
        cudaMalloc(&c->counters, WS_COUNTERS * sizeof(int)) != cudaSuccess ||
        cudaMalloc(&c->dev_err, sizeof(int)) != cudaSuccess || cudaMalloc(&c->sel, WS_SEL_BYTES) != cudaSuccess ||
        cudaMalloc(&c->scores, WS_SCORES_BYTES) != cudaSuccess ||
        cudaMalloc(&c->suf_ws, WS_SUFFIX_BYTES) != cudaSuccess ||
        cudaMalloc(&c->host_stage, PCK_HOST_STAGE_BYTES) != cudaSuccess) {
        cudaGetLastError();
        pck_destroy(c);
        return PCK_ENOMEM;
    }
    cudaMemset(c->counters, 0, WS_COUNTERS * sizeof(int));
    cudaMemset(c->dev_err, 0, sizeof(int));
    if (cudaDeviceSynchronize() != cudaSuccess) {
        pck_destroy(c);
        return PCK_ECUDA;
    }
    *out = c;
    return PCK_OK;
}

void pck_destroy(pck_ctx* c) {
    if (!c) return;
    cudaSetDevice(c->device);
    cudaDeviceSynchronize();
    for (auto& kv : c->slots) free_slot(c, kv.second, nullptr);
    cudaDeviceSynchronize();
    for (auto& r : c->means.freed)
        if (r.ready) cudaEventDestroy(r.ready);
    for (auto& ch : c->means.chunks) cudaFree(ch.base);
    cudaFree(c->partials);
    cudaFree(c->counters);
    cudaFree(c->dev_err);
    cudaFree(c->sel);
    cudaFree(c->scores);
    cudaFree(c->suf_ws);
    cudaFree(c->host_stage);
    delete c;
}

const char* pck_last_error(const pck_ctx* c) { return c ? c->err.c_str() : "no context"; }

int pck_store(pck_ctx* c, const char* sid, int layer, int H_kv, int N, int D, int fmt, const void* K, const void* V,
              int src_dtype, void* stream) {
    if (!c) return PCK_EINVAL;
    if (!sid || !K || !V) return fail(c, PCK_EINVAL, "NULL sid/K/V");
    if (H_kv < 1 || H_kv > PCK_MAX_HEADS || N < 1) return fail(c, PCK_EINVAL, "bad H_kv=%d or N=%d", H_kv, N);
    if (fmt != PCK_FMT_FP16 && fmt != PCK_FMT_MLX4G32) return fail(c, PCK_EINVAL, "fmt=%d", fmt);
    if (!d_ok(D, fmt))
        return fail(c, PCK_EUNSUPPORTED, "D=%d (fp16 slots: 32, 64, 96, 128, 160, 192, 256, 512; mlx4g32: 64, 128, 192, 256)", D);
    if (!dtype_ok(src_dtype)) return fail(c, PCK_EINVAL, "src_dtype=%d", src_dtype);
    if ((reinterpret_cast<uintptr_t>(K) | reinterpret_cast<uintptr_t>(V)) & 15)
        return fail(c, PCK_EINVAL, "K/V must be 16-byte aligned");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int ntiles = (N + TILE_TOK - 1) / TILE_TOK;
    const size_t bytes = static_cast<size_t>(H_kv) * ntiles * tile_bytes(fmt, D);
    uint8_t* tiles = nullptr;
    if (cudaMallocAsync(reinterpret_cast<void**>(&tiles), bytes, st) != cudaSuccess) {
        cudaGetLastError();
        return fail(c, PCK_ENOMEM, "cannot allocate %zu bytes for the slot", bytes);
    }
    cudaError_t e;
    const int f16 = src_dtype == PCK_DT_F16;
    if (fmt == PCK_FMT_FP16) {
        e = launch_relayout_fp16(K, V, f16, H_kv, N, D, ntiles, tiles, st, c->sms);
    } else {
        const int64_t rows = static_cast<int64_t>(H_kv) * N;   // head rows [H_kv * N, D]
        const size_t rec = static_cast<size_t>(D / 2 + D / 8);
        uint8_t* recs = nullptr;
        if (cudaMallocAsync(reinterpret_cast<void**>(&recs), 2 * rec * rows, st) != cudaSuccess) {
            cudaGetLastError();
            cudaFreeAsync(tiles, st);
            return fail(c, PCK_ENOMEM, "cannot allocate the quantiser staging buffer");
        }
        e = launch_quantize(K, f16, rows, D, recs, st, c->sms);
        if (e == cudaSuccess) e = launch_quantize(V, f16, rows, D, recs + rec * rows, st, c->sms);
        if (e == cudaSuccess) e = launch_relayout_mlx4(recs, recs + rec * rows, 1, H_kv, N, D, ntiles, tiles, st, c->sms);
        cudaFreeAsync(recs, st);
    }
    if (e != cudaSuccess) {
        cudaFreeAsync(tiles, st);
        return cuda_fail(c, e, "store launch");
    }
    Slot* s = put_slot(c, key_of(sid, layer), st);
    s->fmt = fmt;
    s->H_kv = H_kv;
    s->N = N;
    s->D = D;
    s->ntiles = ntiles;
    s->tiles = tiles;
    s->bytes = bytes;
    c->bytes_resident += static_cast<int64_t>(bytes);
    ++c->stores;
    return PCK_OK;
}

int pck_store_records(pck_ctx* c, const char* sid, int layer, int H_kv, int N, int D, const void* K_rec,
                      const void* V_rec, void* stream) {
    if (!c) return PCK_EINVAL;
    if (!sid || !K_rec || !V_rec) return fail(c, PCK_EINVAL, "NULL sid/records");
    if (H_kv < 1 || H_kv > PCK_MAX_HEADS || N < 1) return fail(c, PCK_EINVAL, "bad H_kv=%d or N=%d", H_kv, N);
    if (!d_ok(D, PCK_FMT_MLX4G32)) return fail(c, PCK_EUNSUPPORTED, "D=%d (mlx4g32 slots: 64, 128, 192, 256)", D);
    if ((reinterpret_cast<uintptr_t>(K_rec) | reinterpret_cast<uintptr_t>(V_rec)) & 3)
        return fail(c, PCK_EINVAL, "records must be 4-byte aligned");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int ntiles = (N + TILE_TOK - 1) / TILE_TOK;
    const size_t bytes = static_cast<size_t>(H_kv) * ntiles * tile_bytes(PCK_FMT_MLX4G32, D);
    uint8_t* tiles = nullptr;
    if (cudaMallocAsync(reinterpret_cast<void**>(&tiles), bytes, st) != cudaSuccess) {
        cudaGetLastError();
        return fail(c, PCK_ENOMEM, "cannot allocate %zu bytes for the slot", bytes);
    }
    cudaError_t e = launch_relayout_mlx4(K_rec, V_rec, 0, H_kv, N, D, ntiles, tiles, st, c->sms);
    if (e != cudaSuccess) {
        cudaFreeAsync(tiles, st);
        return cuda_fail(c, e, "store_records launch");
    }
    Slot* s = put_slot(c, key_of(sid, layer), st);
    s->fmt = PCK_FMT_MLX4G32;
    s->H_kv = H_kv;
    s->N = N;
    s->D = D;
    s->ntiles = ntiles;
    s->tiles = tiles;
    s->bytes = bytes;
    c->bytes_resident += static_cast<int64_t>(bytes);
    ++c->stores;
    return PCK_OK;
}

int pck_lookup(pck_ctx* c, const char* sid, int layer) {
    if (!c) return PCK_EINVAL;
    if (!sid) return fail(c, PCK_EINVAL, "sid is NULL");
    const std::string k = key_of(sid, layer);
    if (c->slots.count(k)) return PCK_OK;
    return c->cold.count(k) ? PCK_COLDMISS : PCK_MISS;
}

int pck_drop(pck_ctx* c, const char* sid, int layer, void* stream) {
    if (!c) return PCK_EINVAL;
    if (!sid) return fail(c, PCK_EINVAL, "sid is NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int dropped = 0;
    std::vector<std::string> keys;
    if (layer >= 0) {
        keys.push_back(key_of(sid, layer));
    } else {
        const std::string prefix = std::string(sid) + '\x1f';
        for (auto& kv : c->slots)
            if (kv.first.compare(0, prefix.size(), prefix) == 0) keys.push_back(kv.first);
    }
    for (auto& k : keys) {
        auto it = c->slots.find(k);
        if (it == c->slots.end()) continue;
        free_slot(c, it->second, st);
        c->lru.erase(it->second.lru);
        c->slots.erase(it);
        ++dropped;
    }
    return dropped;
}

// The split (fp16 hi + lo, tile layout) copy of a slot's block means, built from the fp32 ones.
static int build_block_means_split(pck_ctx* c, Slot* s, int B, cudaStream_t st) {
    if (s->kmean_split.count(B)) return PCK_OK;
    if (capturing(st)) return fail(c, PCK_EINVAL, "block means are built outside a stream capture");
    const int nb = (s->N + B - 1) / B;
    const size_t bytes = kmean_split_bytes(*s, B);
    uint8_t* out = arena_alloc(c, bytes);
    if (!out) return fail(c, PCK_ENOMEM, "cannot allocate split block means");
    const cudaError_t e = launch_block_means_split(s->kmean[B], s->H_kv, nb, s->D, out, st);
    if (e != cudaSuccess) {
        arena_free(c, out, bytes, st);
        return cuda_fail(c, e, "split block means launch");
    }
    s->kmean_split[B] = out;
    s->bytes += bytes;
    c->bytes_resident += static_cast<int64_t>(bytes);
    return PCK_OK;
}

int pck_build_block_means(pck_ctx* c, const char* sid, int layer, int B, void* stream) {
    if (!c) return PCK_EINVAL;
    Slot* s = nullptr;
    int rc = find_slot(c, sid, layer, &s);
    if (rc != PCK_OK) return rc;
    if (s->fmt != PCK_FMT_FP16) return fail(c, PCK_EUNSUPPORTED, "block means are built for fp16 slots only");
    if (B < 16 || B % 16) return fail(c, PCK_EUNSUPPORTED, "B=%d (must be a positive multiple of 16)", B);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (s->kmean.count(B)) {
        const int nb0 = (s->N + B - 1) / B;
        return sparse_fused_ok(s->D, nb0, 1) ? build_block_means_split(c, s, B, st) : PCK_OK;
    }
    if (capturing(st)) return fail(c, PCK_EINVAL, "block means are built outside a stream capture");
    const int nb = (s->N + B - 1) / B;
    const size_t bytes = kmean_bytes(*s, B);
    float* km = reinterpret_cast<float*>(arena_alloc(c, bytes));
    if (!km) return fail(c, PCK_ENOMEM, "cannot allocate block means");
    cudaError_t e = launch_block_means(s->tiles, s->H_kv, s->N, s->D, s->ntiles, B, km, st, c->sms);
    if (e != cudaSuccess) {
        arena_free(c, km, bytes, st);
        return cuda_fail(c, e, "block means launch");
    }
    s->kmean[B] = km;
    s->bytes += bytes;
    c->bytes_resident += static_cast<int64_t>(bytes);
    // the copy the one-kernel sparse form scores from, where that form applies
    if (sparse_fused_ok(s->D, nb, 1)) return build_block_means_split(c, s, B, st);
    return PCK_OK;
}

static int query_common(pck_ctx* c, const char* sid, int layer, int H_q, int D, int M, int S_suf, int H_kv_arg,
                        int q_dtype, const void* Q, const void* K_suf, const void* V_suf, const int32_t* head_map,
                        int causal, int fa_window, float* O, float* LSE, void* stream) {
    if (!c) return PCK_EINVAL;
    if (!Q || !O) return fail(c, PCK_EINVAL, "NULL Q or O");
    if (reinterpret_cast<uintptr_t>(O) & 15) return fail(c, PCK_EINVAL, "O must be 16-byte aligned");
    if (fa_window < 0) return fail(c, PCK_EINVAL, "fa_window=%d", fa_window);
    if (!dtype_ok(q_dtype)) return fail(c, PCK_EINVAL, "q_dtype=%d", q_dtype);
    if (M < 1) return fail(c, PCK_EINVAL, "M=%d", M);
    if (S_suf < 0) return fail(c, PCK_EINVAL, "S_suf=%d", S_suf);
    if (S_suf > 0 && (!K_suf || !V_suf)) return fail(c, PCK_EINVAL, "S_suf=%d with NULL K_suf/V_suf", S_suf);
    Slot* s = nullptr;
    int rc = find_slot(c, sid, layer, &s);
    if (rc != PCK_OK) return rc;
    if (D != s->D) return fail(c, PCK_EINVAL, "D=%d but the slot holds D=%d", D, s->D);
    if (H_kv_arg > 0 && H_kv_arg != s->H_kv)
        return fail(c, PCK_EINVAL, "H_kv=%d but the slot holds H_kv=%d", H_kv_arg, s->H_kv);
    WorkGroup grp[MAX_GROUPS];
    int n_groups = 0;
    rc = build_groups(c, H_q, s->H_kv, head_map, grp, &n_groups, nullptr, nullptr, d_gmax(D));
    if (rc != PCK_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (M == 1) {
        DescIn d{s, Q, O, LSE, K_suf, V_suf};
        d.window = fa_window;
        rc = run_decode(c, s->fmt, D, H_q, s->H_kv, S_suf, q_dtype == PCK_DT_F16, grp, n_groups, &d, 1, 0, 0, 0, nullptr, st);
        if (rc != PCK_OK) return rc;
        return check_async(c);
    }
    if (q_dtype != PCK_DT_F16) return fail(c, PCK_EUNSUPPORTED, "M>1 needs fp16 Q");
    if (reinterpret_cast<uintptr_t>(Q) & 15) return fail(c, PCK_EINVAL, "Q must be 16-byte aligned");
    if (S_suf > 0 && ((reinterpret_cast<uintptr_t>(K_suf) | reinterpret_cast<uintptr_t>(V_suf)) & 15))
        return fail(c, PCK_EINVAL, "K_suf/V_suf must be 16-byte aligned when M > 1");
    // An mlx4g32 slot is attended as an fp16 slot of head dimension 2D holding [hi | lo] fp16 pairs
    // of its dequantised values (S = [Q | Q] [K_hi | K_lo]^T, O = P V_hi + P V_lo): the tensor-core
    // kernel runs at width DK = 2D.
    const bool split = s->fmt == PCK_FMT_MLX4G32;
    const int DK = split ? 2 * D : D;
    if (!prefill_supported(DK))
        return fail(c, PCK_EUNSUPPORTED, "M>1 kernel not available for D=%d%s", D, split ? " on an mlx4g32 slot" : "");
    if (S_suf > 0 && static_cast<size_t>(s->H_kv) * 2 * fp16_region_bytes((S_suf + TILE_TOK - 1) / TILE_TOK, DK) >
                         WS_SUFFIX_BYTES)
        return fail(c, PCK_EUNSUPPORTED, "suffix of %d tokens exceeds the staging workspace", S_suf);
    const int suf_ntiles = (S_suf + TILE_TOK - 1) / TILE_TOK;
    if (S_suf > 0) {   // stage the suffix in the resident layout (the MMA operand layout)
        // released early: the attention kernel fetches its first resident prefix blocks while this
        // runs, and waits for it before touching the staged suffix
        cudaError_t e = launch_relayout_fp16(K_suf, V_suf, 1, s->H_kv, S_suf, D, suf_ntiles, c->suf_ws, st, c->sms, DK, 1);
        if (e != cudaSuccess) return cuda_fail(c, e, "suffix staging launch");
    }
    uint8_t* kv = s->tiles;
    if (split) {
        const size_t bytes = static_cast<size_t>(s->H_kv) * 2 * fp16_region_bytes(s->ntiles, DK);
        if (cudaMallocAsync(reinterpret_cast<void**>(&kv), bytes, st) != cudaSuccess) {
            cudaGetLastError();
            return fail(c, PCK_ENOMEM, "cannot allocate %zu bytes for the dequantised slot", bytes);
        }
        cudaError_t e = launch_mlx4_split(s->tiles, s->H_kv, s->ntiles, D, kv, st);
        if (e != cudaSuccess) {
            cudaFreeAsync(kv, st);
            return cuda_fail(c, e, "dequantise launch");
        }
    }
    PrefillParams pp{};
    pp.Q = static_cast<const __half*>(Q);
    pp.kv = kv;
    pp.O = O;
    pp.LSE = LSE;
    pp.H_q = H_q;
    pp.H_kv = s->H_kv;
    pp.M = M;
    pp.N = s->N;
    pp.ntiles = s->ntiles;
    pp.S_suf = S_suf;
    pp.causal = causal;
    pp.q_dup = split ? 1 : 0;
    pp.window = fa_window;
    pp.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
    pp.err = c->dev_err;
    cudaError_t e = launch_prefill(pp, grp, n_groups, S_suf > 0 ? c->suf_ws : nullptr, suf_ntiles, c->partials,
                                   WS_PARTIAL_BYTES, c->sms, st, DK);
    if (split) cudaFreeAsync(kv, st);   // stream-ordered: after the kernels that read it
    if (e != cudaSuccess) return cuda_fail(c, e, "prefill launch");
    ++c->queries;
    return check_async(c);
}

int pck_query(pck_ctx* c, const char* sid, int layer, int H_q, int D, int M, int q_dtype, const void* Q,
              const int32_t* head_map, int top_k, int fa_window, float* O, float* LSE, void* stream) {
    if (!c) return PCK_EINVAL;
    Slot* s = nullptr;
    int rc = find_slot(c, sid, layer, &s);
    if (rc != PCK_OK) return rc;
    if (top_k != 0 && top_k < s->N)
        return fail(c, PCK_EUNSUPPORTED, "top_k=%d < N=%d (only 0 or >= N, i.e. dense, is defined)", top_k, s->N);
    return query_common(c, sid, layer, H_q, D, M, 0, 0, q_dtype, Q, nullptr, nullptr, head_map, 1, fa_window, O, LSE,
                        stream);
}

int pck_query_fused(pck_ctx* c, const char* sid, int layer, int H_q, int D, int M, int S_suf, int H_kv, int q_dtype,
                    const void* Q, const void* K_suf, const void* V_suf, const int32_t* head_map, int causal,
                    int fa_window, float* O, float* LSE, void* stream) {
    if (!c) return PCK_EINVAL;
    if (H_kv < 1) return fail(c, PCK_EINVAL, "H_kv=%d", H_kv);
    return query_common(c, sid, layer, H_q, D, M, S_suf, H_kv, q_dtype, Q, K_suf, V_suf, head_map, causal, fa_window,
                        O, LSE, stream);
}

// One sparse query: its slot, Q, outputs, suffix and (optional) index output.
struct SparseIn {
    const char* sid;
    int layer;
    const void* Q;
    float* O;
    float* LSE;
    const void* K_suf;
    const void* V_suf;
    int32_t* idx_out;
};

// n sparse queries of the same shapes (slots with the same N): block scoring of all of them in one
// launch, their top-K selections in one launch, then one split-K gather decode (+ merge) over the
// selected tiles of all of them.
static int sparse_run(pck_ctx* c, int n, const SparseIn* q, int H_q, int D, int B, int K_top, int H_kv, int S_suf,
                      int q_dtype, const int32_t* head_map, int fa_window, void* stream) {
    if (!c) return PCK_EINVAL;
    if (n < 1 || n > MAX_DESC) return fail(c, PCK_EINVAL, "n=%d (1..%d queries per call)", n, MAX_DESC);
    if (fa_window != 0) return fail(c, PCK_EUNSUPPORTED, "fa_window=%d (only 0 is defined)", fa_window);
    if (!dtype_ok(q_dtype)) return fail(c, PCK_EINVAL, "q_dtype=%d", q_dtype);
    if (K_top < 1) return fail(c, PCK_EINVAL, "K_top=%d", K_top);
    if (S_suf < 0) return fail(c, PCK_EINVAL, "S_suf=%d", S_suf);
    if (B < 16 || B % 16) return fail(c, PCK_EUNSUPPORTED, "B=%d (must be a positive multiple of 16)", B);
    if (D != 64 && D != 128 && D != 256) return fail(c, PCK_EUNSUPPORTED, "D=%d (sparse queries take 64, 128 or 256)", D);
    Slot* slots[MAX_DESC];
    for (int i = 0; i < n; ++i) {
        if (!q[i].Q || !q[i].O) return fail(c, PCK_EINVAL, "query %d: NULL Q or O", i);
        if ((reinterpret_cast<uintptr_t>(q[i].O) | reinterpret_cast<uintptr_t>(q[i].Q)) & 15)
            return fail(c, PCK_EINVAL, "query %d: Q and O must be 16-byte aligned", i);
        if (S_suf > 0 && (!q[i].K_suf || !q[i].V_suf)) return fail(c, PCK_EINVAL, "query %d: bad suffix arguments", i);
        int rc = find_slot(c, q[i].sid, q[i].layer, &slots[i]);
        if (rc != PCK_OK) return rc;
        const Slot* s = slots[i];
        if (D != s->D) return fail(c, PCK_EINVAL, "query %d: D=%d but the slot holds D=%d", i, D, s->D);
        if (H_kv != s->H_kv) return fail(c, PCK_EINVAL, "query %d: H_kv=%d but the slot holds H_kv=%d", i, H_kv, s->H_kv);
        if (s->fmt != PCK_FMT_FP16) return fail(c, PCK_EUNSUPPORTED, "sparse queries need an fp16 slot");
        if (s->N != slots[0]->N) return fail(c, PCK_EUNSUPPORTED, "query %d: N=%d differs from N=%d", i, s->N, slots[0]->N);
    }
    const int nb = (slots[0]->N + B - 1) / B;
    const int K_eff = std::min(K_top, nb);
    if (K_eff > 64) return fail(c, PCK_EUNSUPPORTED, "K_top=%d (at most 64)", K_top);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    for (int i = 0; i < n; ++i) {   // cached per (slot, B): only the first query of a slot builds them
        int rc = pck_build_block_means(c, q[i].sid, q[i].layer, B, stream);
        if (rc != PCK_OK) return rc;
    }
    bool suf_aligned = true;   // the fused kernel copies suffix rows with the bulk-copy engine
    for (int i = 0; i < n && S_suf > 0; ++i)
        suf_aligned = suf_aligned && !((reinterpret_cast<uintptr_t>(q[i].K_suf) | reinterpret_cast<uintptr_t>(q[i].V_suf)) & 15);
    // The fused kernel runs a CTA per work item; with few items its per-CTA streaming rate bounds
    // the call, and the four-kernel form (which spreads every phase over all SMs) is faster.
    constexpr int FUSED_MIN_ITEMS = 32;
    int n_items_est = 0;
    {
        int hm_cnt[PCK_MAX_HEADS] = {};
        for (int h = 0; h < H_q; ++h) {
            const int gk = head_map ? head_map[h] : (H_q % H_kv ? 0 : h / (H_q / H_kv));
            if (gk >= 0 && gk < PCK_MAX_HEADS) ++hm_cnt[gk];
        }
        const int gm = sparse_fused_gmax(D);
        for (int gk = 0; gk < H_kv && gk < PCK_MAX_HEADS; ++gk) n_items_est += n * ((hm_cnt[gk] + gm - 1) / gm);
    }
    if (suf_aligned && n_items_est >= FUSED_MIN_ITEMS && sparse_fused_ok(D, nb, K_eff)) {
        // the whole query in one kernel, a CTA per work item
        for (int i = 0; i < n; ++i) {
            const int rc = build_block_means_split(c, slots[i], B, st);
            if (rc != PCK_OK) return rc;
        }
        static thread_local FusedSparseParams fp;
        std::memset(&fp, 0, sizeof fp);
        int n_groups = 0, max_nq = 0;
        int rc = build_groups(c, H_q, H_kv, head_map, fp.grp, &n_groups, nullptr, &max_nq, sparse_fused_gmax(D));
        if (rc != PCK_OK) return rc;
        fp.n_sess = n;
        fp.n_groups = n_groups;
        fp.H_q = H_q;
        fp.D = D;
        fp.N = slots[0]->N;
        fp.ntiles = slots[0]->ntiles;
        fp.nb = nb;
        fp.tpb = B / 16;
        fp.K_eff = K_eff;
        fp.S_suf = S_suf;
        fp.q_f16 = q_dtype == PCK_DT_F16;
        fp.tau = static_cast<float>(1.0 / std::sqrt(static_cast<double>(D)));
        fp.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
        fp.err = c->dev_err;
        for (int i = 0; i < n; ++i)
            fp.sess[i] = FusedSession{slots[i]->kmean_split[B], q[i].Q, slots[i]->tiles,
                                      static_cast<const __half*>(q[i].K_suf), static_cast<const __half*>(q[i].V_suf),
                                      q[i].O, q[i].LSE, q[i].idx_out};
        const cudaError_t e = launch_sparse_fused(fp, max_nq, st);
        if (e != cudaSuccess) return cuda_fail(c, e, "sparse launch");
        return check_async(c);
    }
    static thread_local SelectParams sp;
    std::memset(&sp, 0, sizeof sp);
    int n_groups = 0, max_nq = 0;
    int rc = build_groups(c, H_q, H_kv, head_map, sp.grp, &n_groups, sp.head_map, &max_nq);
    if (rc != PCK_OK) return rc;
    const int sel_max = max_nq * K_eff;
    const size_t lists = static_cast<size_t>(n_groups) * sel_max;   // entries per query
    const int n_items = n * n_groups;
    // selection workspace: block lists, q-head masks, then the items' unit counts and offsets
    const size_t cnt_off = (static_cast<size_t>(n) * lists * (sizeof(int) + 1) + 15) & ~size_t(15);
    const size_t base_off = cnt_off + static_cast<size_t>(n_items) * sizeof(int);
    if (base_off + static_cast<size_t>(n_items + 1) * sizeof(int) > WS_SEL_BYTES)
        return fail(c, PCK_EUNSUPPORTED, "selection lists too large");
    if (static_cast<size_t>(n) * H_q * nb * sizeof(float) > WS_SCORES_BYTES)
        return fail(c, PCK_EUNSUPPORTED, "too many blocks for the score workspace");
    int* sel_blocks = reinterpret_cast<int*>(c->sel);
    uint8_t* sel_mask = c->sel + static_cast<size_t>(n) * lists * sizeof(int);
    int* item_cnt = reinterpret_cast<int*>(c->sel + cnt_off);
    int* item_base = reinterpret_cast<int*>(c->sel + base_off);
    sp.q_f16 = q_dtype == PCK_DT_F16;
    sp.H_q = H_q;
    sp.H_kv = H_kv;
    sp.D = D;
    sp.nb = nb;
    sp.K_top = K_top;
    sp.K_eff = K_eff;
    sp.sel_max = sel_max;
    sp.n_groups = n_groups;
    sp.n_sess = n;
    sp.tau = static_cast<float>(1.0 / std::sqrt(static_cast<double>(D)));
    sp.tpb = B / 16;
    sp.ntiles = slots[0]->ntiles;
    sp.item_cnt = item_cnt;
    sp.item_base = item_base;
    sp.done = reinterpret_cast<unsigned*>(c->counters + (WS_COUNTERS - 1));   // items selected so far
    sp.err = c->dev_err;
    static thread_local DescIn d[MAX_DESC];
    for (int i = 0; i < n; ++i) {
        SelSession& ss = sp.sess[i];
        ss.kmean = slots[i]->kmean[B];
        ss.Q = q[i].Q;
        ss.scores = c->scores + static_cast<size_t>(i) * H_q * nb;
        ss.idx_out = q[i].idx_out;
        ss.sel_blocks = sel_blocks + i * lists;
        ss.sel_mask = sel_mask + i * lists;
        d[i] = DescIn{slots[i], q[i].Q, q[i].O, q[i].LSE, q[i].K_suf, q[i].V_suf, ss.sel_blocks, ss.sel_mask};
    }
    cudaError_t e = launch_select(sp, st, c->sms);
    if (e != cudaSuccess) return cuda_fail(c, e, "selector launch");
    rc = run_decode(c, PCK_FMT_FP16, D, H_q, H_kv, S_suf, q_dtype == PCK_DT_F16, sp.grp, n_groups, d, n, 1, B / 16,
                    sel_max, item_base, st);
    if (rc != PCK_OK) return rc;
    return check_async(c);
}

int pck_query_sparse_auto(pck_ctx* c, const char* sid, int layer, int H_q, int D, int B, int K_top, int H_kv,
                          int q_dtype, const void* Q, const int32_t* head_map, int fa_window, float* O, float* LSE,
                          int32_t* idx_out, void* stream) {
    const SparseIn q{sid, layer, Q, O, LSE, nullptr, nullptr, idx_out};
    return sparse_run(c, 1, &q, H_q, D, B, K_top, H_kv, 0, q_dtype, head_map, fa_window, stream);
}

int pck_query_sparse_auto_fused(pck_ctx* c, const char* sid, int layer, int H_q, int D, int B, int K_top, int H_kv,
                                int S_suf, int q_dtype, const void* Q, const void* K_suf, const void* V_suf,
                                const int32_t* head_map, int fa_window, float* O, float* LSE, int32_t* idx_out,
                                void* stream) {
    const SparseIn q{sid, layer, Q, O, LSE, K_suf, V_suf, idx_out};
    return sparse_run(c, 1, &q, H_q, D, B, K_top, H_kv, S_suf, q_dtype, head_map, fa_window, stream);
}

int pck_query_sparse_batch(pck_ctx* c, int n, const pck_sparse_desc* descs, int H_q, int H_kv, int D, int B,
                           int K_top, int S_suf, int q_dtype, const int32_t* head_map, void* stream) {
    if (!c) return PCK_EINVAL;
    if (n < 1 || n > PCK_MAX_BATCH || !descs) return fail(c, PCK_EINVAL, "n=%d (1..%d) or NULL descs", n, PCK_MAX_BATCH);
    SparseIn q[PCK_MAX_BATCH];
    for (int i = 0; i < n; ++i)
        q[i] = SparseIn{descs[i].sid, descs[i].layer, descs[i].Q, descs[i].O, descs[i].LSE,
                        S_suf > 0 ? descs[i].K_suf : nullptr, S_suf > 0 ? descs[i].V_suf : nullptr, descs[i].idx_out};
    return sparse_run(c, n, q, H_q, D, B, K_top, H_kv, S_suf, q_dtype, head_map, 0, stream);
}

int pck_query_batch(pck_ctx* c, int n, const pck_query_desc* descs, int H_q, int H_kv, int D, int S_suf, int q_dtype,
                    const int32_t* head_map, void* stream) {
    if (!c) return PCK_EINVAL;
    if (n < 1 || n > PCK_MAX_BATCH || !descs) return fail(c, PCK_EINVAL, "n=%d (1..%d) or NULL descs", n, PCK_MAX_BATCH);
    if (!dtype_ok(q_dtype)) return fail(c, PCK_EINVAL, "q_dtype=%d", q_dtype);
    if (S_suf < 0) return fail(c, PCK_EINVAL, "S_suf=%d", S_suf);
    DescIn ds[PCK_MAX_BATCH];
    int fmt = -1;
    for (int i = 0; i < n; ++i) {
        Slot* s = nullptr;
        int rc = find_slot(c, descs[i].sid, descs[i].layer, &s);
        if (rc != PCK_OK) return rc;
        if (s->D != D || s->H_kv != H_kv)
            return fail(c, PCK_EINVAL, "descriptor %d: slot shape (H_kv=%d, D=%d) differs from the batch", i, s->H_kv, s->D);
        if (fmt >= 0 && s->fmt != fmt) return fail(c, PCK_EINVAL, "descriptor %d: mixed slot formats", i);
        fmt = s->fmt;
        if (!descs[i].Q || !descs[i].O) return fail(c, PCK_EINVAL, "descriptor %d: NULL Q or O", i);
        if ((reinterpret_cast<uintptr_t>(descs[i].O) | reinterpret_cast<uintptr_t>(descs[i].Q)) & 15)
            return fail(c, PCK_EINVAL, "descriptor %d: Q and O must be 16-byte aligned", i);
        if (S_suf > 0 && (!descs[i].K_suf || !descs[i].V_suf))
            return fail(c, PCK_EINVAL, "descriptor %d: NULL suffix", i);
        ds[i] = DescIn{s, descs[i].Q, descs[i].O, descs[i].LSE, descs[i].K_suf, descs[i].V_suf};
    }
    WorkGroup grp[MAX_GROUPS];
    int n_groups = 0;
    int rc = build_groups(c, H_q, H_kv, head_map, grp, &n_groups, nullptr, nullptr, d_gmax(D));
    if (rc != PCK_OK) return rc;
    rc = run_decode(c, fmt, D, H_q, H_kv, S_suf, q_dtype == PCK_DT_F16, grp, n_groups, ds, n, 0, 0, 0, nullptr,
                    static_cast<cudaStream_t>(stream));
    if (rc != PCK_OK) return rc;
    return check_async(c);
}

// The device-side address of page-locked host memory (nullptr when p is not such memory).
static void* host_device_ptr(const void* p) {
    cudaPointerAttributes a;
    if (!p || cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

int pck_query_batch_host(pck_ctx* c, int n, const pck_query_desc* descs, int H_q, int H_kv, int D, int S_suf,
                         int q_dtype, const int32_t* head_map, void* stream) {
    if (!c) return PCK_EINVAL;
    if (n < 1 || n > PCK_MAX_BATCH || !descs) return fail(c, PCK_EINVAL, "n=%d (1..%d) or NULL descs", n, PCK_MAX_BATCH);
    if (!dtype_ok(q_dtype)) return fail(c, PCK_EINVAL, "q_dtype=%d", q_dtype);
    if (S_suf < 0) return fail(c, PCK_EINVAL, "S_suf=%d", S_suf);
    if (H_q < 1 || H_q > PCK_MAX_HEADS || H_kv < 1 || H_kv > PCK_MAX_HEADS || D < 1 || D > 512)
        return fail(c, PCK_EINVAL, "H_q=%d H_kv=%d D=%d", H_q, H_kv, D);
    const size_t q_bytes = static_cast<size_t>(H_q) * D * (q_dtype == PCK_DT_F16 ? 2 : 4);
    const size_t s_bytes = static_cast<size_t>(H_kv) * S_suf * D * 2;
    auto al16 = [](size_t x) { return (x + 15) & ~size_t(15); };
    const size_t per = al16(q_bytes) + 2 * al16(s_bytes);
    if (per * n > PCK_HOST_STAGE_BYTES)
        return fail(c, PCK_EUNSUPPORTED, "%zu bytes of inputs (the staging memory holds %u)", per * n, PCK_HOST_STAGE_BYTES);
    if ((q_bytes | s_bytes) & 15) return fail(c, PCK_EINVAL, "Q and suffix sizes must be multiples of 16 bytes");
    static thread_local CopySegs segs;
    static thread_local pck_query_desc dd[PCK_MAX_BATCH];
    segs.n = 0;
    auto add = [&](const void* host, uint8_t* dst, size_t bytes, const char* what, int i) -> int {
        void* src = host_device_ptr(host);
        if (!src) return fail(c, PCK_EINVAL, "descriptor %d: %s is not page-locked host memory", i, what);
        if (reinterpret_cast<uintptr_t>(src) & 15) return fail(c, PCK_EINVAL, "descriptor %d: %s not 16-byte aligned", i, what);
        segs.src[segs.n] = src;
        segs.dst[segs.n] = dst;
        segs.n16[segs.n] = static_cast<int>(bytes / 16);
        ++segs.n;
        return PCK_OK;
    };
    for (int i = 0; i < n; ++i) {
        uint8_t* base = c->host_stage + per * i;
        dd[i] = descs[i];
        int rc = add(descs[i].Q, base, q_bytes, "Q", i);
        if (rc != PCK_OK) return rc;
        dd[i].Q = base;
        if (S_suf > 0) {
            rc = add(descs[i].K_suf, base + al16(q_bytes), s_bytes, "K_suf", i);
            if (rc != PCK_OK) return rc;
            rc = add(descs[i].V_suf, base + al16(q_bytes) + al16(s_bytes), s_bytes, "V_suf", i);
            if (rc != PCK_OK) return rc;
            dd[i].K_suf = base + al16(q_bytes);
            dd[i].V_suf = base + al16(q_bytes) + al16(s_bytes);
        }
        dd[i].O = static_cast<float*>(host_device_ptr(descs[i].O));
        if (!dd[i].O) return fail(c, PCK_EINVAL, "descriptor %d: O is not page-locked host memory", i);
        if (descs[i].LSE) {
            dd[i].LSE = static_cast<float*>(host_device_ptr(descs[i].LSE));
            if (!dd[i].LSE) return fail(c, PCK_EINVAL, "descriptor %d: LSE is not page-locked host memory", i);
        }
    }
    const cudaError_t e = launch_copy_segments(segs, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(c, e, "staging copy");
    return pck_query_batch(c, n, dd, H_q, H_kv, D, S_suf, q_dtype, head_map, stream);
}

int pck_query_sparse(pck_ctx* c, const char* sid, int layer, int H_q, int D, int K_sparse_max, int q_dtype,
                     const void* Q, const int32_t* indices, const int32_t* counts, const int32_t* head_map, int fa_window,
                     float* O, float* LSE, void* stream) {
    if (!c) return PCK_EINVAL;
    if (!Q || !O || !indices || !counts) return fail(c, PCK_EINVAL, "NULL Q, O, indices or counts");
    if ((reinterpret_cast<uintptr_t>(O) | reinterpret_cast<uintptr_t>(Q)) & 15)
        return fail(c, PCK_EINVAL, "Q and O must be 16-byte aligned");
    if (fa_window != 0) return fail(c, PCK_EUNSUPPORTED, "fa_window=%d (only 0 is defined)", fa_window);
    if (!dtype_ok(q_dtype)) return fail(c, PCK_EINVAL, "q_dtype=%d", q_dtype);
    if (K_sparse_max < 1) return fail(c, PCK_EINVAL, "K_sparse_max=%d", K_sparse_max);
    if (H_q < 1 || H_q > MAX_DESC) return fail(c, PCK_EINVAL, "H_q=%d (1..%d)", H_q, MAX_DESC);
    Slot* s = nullptr;
    int rc = find_slot(c, sid, layer, &s);
    if (rc != PCK_OK) return rc;
    if (s->fmt != PCK_FMT_FP16) return fail(c, PCK_EUNSUPPORTED, "QUERY_SPARSE needs an fp16 slot");
    if (D != s->D) return fail(c, PCK_EINVAL, "D=%d but the slot holds D=%d", D, s->D);
    int8_t hm[PCK_MAX_HEADS];
    WorkGroup grp_all[MAX_GROUPS];
    int n_groups_all = 0;
    rc = build_groups(c, H_q, s->H_kv, head_map, grp_all, &n_groups_all, hm, nullptr);
    if (rc != PCK_OK) return rc;
    // every head's list: 1 <= counts[h] <= K_sparse_max strictly ascending positions in [0, N)
    int kmax = 0;
    for (int h = 0; h < H_q; ++h) {
        const int n = counts[h];
        if (n < 1 || n > K_sparse_max) return fail(c, PCK_EINVAL, "counts[%d]=%d outside [1, %d]", h, n, K_sparse_max);
        const int32_t* row = indices + static_cast<size_t>(h) * K_sparse_max;
        for (int k = 0; k < n; ++k) {
            if (row[k] < 0 || row[k] >= s->N)
                return fail(c, PCK_EINVAL, "indices[%d][%d]=%d outside [0, %d)", h, k, row[k], s->N);
            if (k > 0 && row[k] <= row[k - 1])
                return fail(c, PCK_EINVAL, "indices[%d] not strictly ascending at %d (duplicate or unsorted)", h, k);
        }
        kmax = std::max(kmax, n);
    }
    // one device buffer: index rows [H_q][kmax], counts [H_q], head map [H_q] (int8), then one
    // compact fp16 slot per q head holding its gathered tokens
    const int ntmax = (kmax + TILE_TOK - 1) / TILE_TOK;
    const size_t head_stride = 2 * fp16_region_bytes(ntmax, D);
    const size_t meta = (static_cast<size_t>(H_q) * (kmax + 1) * sizeof(int32_t) + H_q + 255) & ~size_t(255);
    std::vector<uint8_t> host(meta, 0);
    int32_t* hidx = reinterpret_cast<int32_t*>(host.data());
    for (int h = 0; h < H_q; ++h)
        std::memcpy(hidx + static_cast<size_t>(h) * kmax, indices + static_cast<size_t>(h) * K_sparse_max,
                    sizeof(int32_t) * counts[h]);
    std::memcpy(hidx + static_cast<size_t>(H_q) * kmax, counts, sizeof(int32_t) * H_q);
    std::memcpy(host.data() + static_cast<size_t>(H_q) * (kmax + 1) * sizeof(int32_t), hm, H_q);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* buf = nullptr;
    const size_t bytes = meta + static_cast<size_t>(H_q) * head_stride;
    if (cudaMallocAsync(reinterpret_cast<void**>(&buf), bytes, st) != cudaSuccess) {
        cudaGetLastError();
        return fail(c, PCK_ENOMEM, "cannot allocate %zu bytes for the gathered tokens", bytes);
    }
    cudaError_t e = cudaMemcpyAsync(buf, host.data(), meta, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) {
        const int32_t* didx = reinterpret_cast<const int32_t*>(buf);
        e = launch_gather_fp16(s->tiles, s->ntiles, D, didx, didx + static_cast<size_t>(H_q) * kmax,
                               reinterpret_cast<const int8_t*>(buf + static_cast<size_t>(H_q) * (kmax + 1) * sizeof(int32_t)),
                               H_q, kmax, head_stride, buf + meta, st);
    }
    if (e != cudaSuccess) {
        cudaFreeAsync(buf, st);
        return cuda_fail(c, e, "gather launch");
    }
    // one dense decode over H_q single-head compact slots (one descriptor per q head)
    Slot tmp[MAX_DESC];
    DescIn d[MAX_DESC];
    const size_t qbytes = static_cast<size_t>(D) * (q_dtype == PCK_DT_F16 ? 2 : 4);
    for (int h = 0; h < H_q; ++h) {
        tmp[h].fmt = PCK_FMT_FP16;
        tmp[h].H_kv = 1;
        tmp[h].N = counts[h];
        tmp[h].D = D;
        tmp[h].ntiles = (counts[h] + TILE_TOK - 1) / TILE_TOK;
        tmp[h].tiles = buf + meta + static_cast<size_t>(h) * head_stride;
        d[h] = DescIn{&tmp[h], static_cast<const uint8_t*>(Q) + h * qbytes, O + static_cast<size_t>(h) * D,
                      LSE ? LSE + h : nullptr, nullptr, nullptr};
    }
    const WorkGroup one{0, 1, {0, -1, -1, -1, -1, -1, -1, -1}};
    rc = run_decode(c, PCK_FMT_FP16, D, 1, 1, 0, q_dtype == PCK_DT_F16, &one, 1, d, H_q, 0, 0, 0, nullptr, st);
    cudaFreeAsync(buf, st);   // stream-ordered: after the kernels that read it
    if (rc != PCK_OK) return rc;
    return check_async(c);
}

int pck_get_block_means(pck_ctx* c, const char* sid, int layer, int B, float* out, void* stream) {
    if (!c) return PCK_EINVAL;
    if (!out) return fail(c, PCK_EINVAL, "NULL out");
    int rc = pck_build_block_means(c, sid, layer, B, stream);
    if (rc != PCK_OK) return rc;
    Slot* s = nullptr;
    rc = find_slot(c, sid, layer, &s);
    if (rc != PCK_OK) return rc;
    const size_t bytes = static_cast<size_t>(s->H_kv) * ((s->N + B - 1) / B) * s->D * sizeof(float);
    cudaError_t e = cudaMemcpyAsync(out, s->kmean[B], bytes, cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(c, e, "block means copy");
    return PCK_OK;
}

int pck_dequantize_mlx4g32(const void* records, int64_t N, int H_kv, int D, int out_dtype, void* out, void* stream) {
    if (!records || !out || N < 0 || H_kv < 1 || H_kv > PCK_MAX_HEADS || D < 8 || D % 8 || (H_kv * D) % 32)
        return PCK_EINVAL;
    if (!dtype_ok(out_dtype)) return PCK_EINVAL;
    if (reinterpret_cast<uintptr_t>(records) & 3) return PCK_EINVAL;
    if (reinterpret_cast<uintptr_t>(out) & 15) return PCK_EINVAL;
    if (N == 0) return PCK_OK;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaError_t e = launch_dequant_records(records, N, H_kv, D, out_dtype == PCK_DT_F16, out,
                                           static_cast<cudaStream_t>(stream), sms > 0 ? sms : 1);
    return e == cudaSuccess ? PCK_OK : PCK_ECUDA;
}

int pck_quantize_mlx4g32(const void* X, int src_dtype, int64_t rows, int kv_dim, void* out_records, void* stream) {
    if (!X || !out_records || rows < 0 || kv_dim < 32 || kv_dim % 32) return PCK_EINVAL;
    if (!dtype_ok(src_dtype)) return PCK_EINVAL;
    if (reinterpret_cast<uintptr_t>(X) & 15) return PCK_EINVAL;
    if (reinterpret_cast<uintptr_t>(out_records) & 3) return PCK_EINVAL;
    if (rows == 0) return PCK_OK;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaError_t e = launch_quantize(X, src_dtype == PCK_DT_F16, rows, kv_dim, out_records,
                                    static_cast<cudaStream_t>(stream), sms > 0 ? sms : 1);
    return e == cudaSuccess ? PCK_OK : PCK_ECUDA;
}

int pck_info(pck_ctx* c, pck_info_t* out) {
    if (!c || !out) return PCK_EINVAL;
    out->slots_used = static_cast<int64_t>(c->slots.size());
    out->slots_max = c->max_slots;
    out->cold_entries = static_cast<int64_t>(c->cold.size());
    out->bytes_resident = c->bytes_resident;
    out->queries_served = c->queries;
    out->stores = c->stores;
    out->evictions = c->evictions;
    return PCK_OK;
}

int pck_sync(pck_ctx* c, void* stream) {
    if (!c) return PCK_EINVAL;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(c, e, "stream synchronize");
    int herr = 0;
    e = cudaMemcpy(&herr, c->dev_err, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(c, e, "error word read");
    if (herr) {
        cudaMemset(c->dev_err, 0, sizeof(int));
        cudaMemset(c->counters, 0, WS_COUNTERS * sizeof(int));
        cudaDeviceSynchronize();
        return fail(c, PCK_ECUDA, "a device wait gave up (code %d); results of the affected calls are invalid", herr);
    }
    return PCK_OK;
}

}  // extern "C"
