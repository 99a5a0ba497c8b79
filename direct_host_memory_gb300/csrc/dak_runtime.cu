// Runtime of the direct-access library: status word, placement of operands across the
// host and HBM tiers, the persistent-grid split between tiers, tier bandwidth probes and
// the prefetch baseline's copy.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstring>
#include <cstdlib>
#include <mutex>
#include <string>
#include <vector>

#include "dak_device.cuh"

namespace dak {

__device__ DevStatus g_status_block = {0, 0, 0ull};

unsigned long long current_context_id() {
    using GetCurrentFn = CUresult (*)(CUcontext*);
    using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* a = nullptr;
        void* b = nullptr;
        cudaDriverEntryPointQueryResult qa, qb;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) == cudaSuccess &&
            qa == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) == cudaSuccess &&
            qb == cudaDriverEntryPointSuccess) {
            get_current = reinterpret_cast<GetCurrentFn>(a);
            get_id = reinterpret_cast<GetIdFn>(b);
        }
        cudaGetLastError();
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

DevStatus* status_ptr() {
    static DevStatus* cache[64] = {nullptr};
    static unsigned long long ctx[64] = {0};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long id = current_context_id();
    if (!cache[dev] || ctx[dev] != id) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_status_block) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        cache[dev] = static_cast<DevStatus*>(ptr);
        ctx[dev] = current_context_id();  // the lookup may have created the context
    }
    return cache[dev];
}

// ------------------------------------------------------------------------------------
// host-link handoff sequences of the public calls (dak_link_begin, dak_tuning.link): a
// device count per slot, and per device and slot the signals of the sequence's launches so
// far (the `after` of its next launch)
// ------------------------------------------------------------------------------------
__device__ unsigned g_link_count[kLinkSlots];
static std::mutex g_link_mu;
static unsigned g_link_after[64][kLinkSlots];

// The device counts of the current device (called with g_link_mu held). A new context (after
// cudaDeviceReset) starts with the module's counts at zero, so the host-side counts of its
// sequences restart too.
static unsigned* link_counts() {
    static unsigned* cache[64] = {nullptr};
    static unsigned long long ctx[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    const unsigned long long id = current_context_id();
    if (!cache[dev] || ctx[dev] != id) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_link_count) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        cache[dev] = static_cast<unsigned*>(ptr);
        ctx[dev] = current_context_id();
        for (int k = 0; k < kLinkSlots; ++k) g_link_after[dev][k] = 0;
    }
    return cache[dev];
}

bool link_join(const dak_tuning* t, LinkHandoff* lk) {
    if (!t || t->link < 1 || t->link > kLinkSlots) return false;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lock(g_link_mu);
    unsigned* c = link_counts();
    if (!c) return false;
    lk->ctr = c + (t->link - 1);
    lk->after = g_link_after[dev][t->link - 1];
    return true;
}

void link_commit(const dak_tuning* t, int signals) {
    int dev = 0;
    if (!t || t->link < 1 || t->link > kLinkSlots || signals <= 0) return;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return;
    std::lock_guard<std::mutex> lock(g_link_mu);
    g_link_after[dev][t->link - 1] += static_cast<unsigned>(signals);
}

}  // namespace dak

extern "C" dak_status dak_link_begin(int slot, void* stream) {
    using namespace dak;
    if (slot < 1 || slot > kLinkSlots) return DAK_ERR_INVALID;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DAK_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_link_mu);
    unsigned* c = link_counts();
    if (!c) return DAK_ERR_CUDA;
    const cudaError_t e = cudaMemsetAsync(c + (slot - 1), 0, sizeof(unsigned), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_status(e);
    g_link_after[dev][slot - 1] = 0;
    return DAK_OK;
}

namespace dak {

// ------------------------------------------------------------------------------------
// allocations: live counts and host-side fault injection
// ------------------------------------------------------------------------------------
static std::atomic<long long> g_live_host{0}, g_live_dev{0};
constexpr int kFaultKinds = 4;  // DAK_FAULT_HOST_ALLOC .. DAK_FAULT_TENSOR_MAP are 1..3
static std::mutex g_fault_mu;
static int g_fault_skip[kFaultKinds], g_fault_count[kFaultKinds];

// DAK_FAULT_INJECT="host_alloc=SKIP:COUNT,device_alloc=COUNT,tensor_map=..." (SKIP defaults
// to 0, COUNT -1 = every call), read once, at the library's first allocation or fault query.
static void load_fault_env() {
    static std::once_flag once;
    std::call_once(once, [] {
        const char* env = std::getenv("DAK_FAULT_INJECT");
        if (!env) return;
        static const char* names[kFaultKinds] = {"", "host_alloc", "device_alloc", "tensor_map"};
        std::string spec(env);
        size_t pos = 0;
        std::lock_guard<std::mutex> lock(g_fault_mu);
        while (pos < spec.size()) {
            size_t end = spec.find(',', pos);
            if (end == std::string::npos) end = spec.size();
            const std::string item = spec.substr(pos, end - pos);
            pos = end + 1;
            const size_t eq = item.find('=');
            if (eq == std::string::npos) continue;
            const std::string name = item.substr(0, eq), val = item.substr(eq + 1);
            for (int k = 1; k < kFaultKinds; ++k) {
                if (name != names[k]) continue;
                const size_t colon = val.find(':');
                const int skip = colon == std::string::npos ? 0 : std::atoi(val.substr(0, colon).c_str());
                const int count = std::atoi(colon == std::string::npos ? val.c_str() : val.substr(colon + 1).c_str());
                g_fault_skip[k] = std::max(0, skip);
                g_fault_count[k] = count;
            }
        }
    });
}

bool fault_due(int kind) {
    if (kind < 1 || kind >= kFaultKinds) return false;
    load_fault_env();
    std::lock_guard<std::mutex> lock(g_fault_mu);
    if (g_fault_count[kind] == 0) return false;
    if (g_fault_skip[kind] > 0) {
        --g_fault_skip[kind];
        return false;
    }
    if (g_fault_count[kind] > 0) --g_fault_count[kind];
    return true;
}

cudaError_t host_alloc_mapped(void** p, size_t bytes) {
    *p = nullptr;
    if (fault_due(DAK_FAULT_HOST_ALLOC)) return cudaErrorMemoryAllocation;
    const cudaError_t e = cudaHostAlloc(p, bytes, cudaHostAllocMapped | cudaHostAllocPortable);
    if (e == cudaSuccess) {
        ++g_live_host;
    } else {
        *p = nullptr;
    }
    return e;
}

void host_free(void* p) {
    if (!p) return;
    cudaFreeHost(p);
    --g_live_host;
}

cudaError_t dev_alloc(void** p, size_t bytes) {
    *p = nullptr;
    if (fault_due(DAK_FAULT_DEVICE_ALLOC)) return cudaErrorMemoryAllocation;
    const cudaError_t e = cudaMalloc(p, bytes);
    if (e == cudaSuccess) {
        ++g_live_dev;
    } else {
        *p = nullptr;
    }
    return e;
}

void dev_free(void* p) {
    if (!p) return;
    cudaFree(p);
    --g_live_dev;
}

dak_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return DAK_OK;
    if (e == cudaErrorMemoryAllocation) return DAK_ERR_DEVICE_ALLOC;
    return DAK_ERR_CUDA;
}

int device_sm_count() {
    static std::atomic<int> cache[64];  // 0 = not looked up yet
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (!n) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = 1;
        }
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

static int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

Sched schedule(int host_units, int hbm_units, int sm_slots, const dak_tuning* t, int default_host_ctas,
               int default_host_window, int default_hbm_window, int max_window) {
    Sched s{};
    int cap = (t && t->host_ctas > 0) ? t->host_ctas : default_host_ctas;
    if (!(t && t->host_ctas > 0) && host_units > 0) {
        // at least the host units' share of the slots: when units are compute-heavy the host
        // side needs its share of SMs, and on this GPU more host CTAs do not congest HBM
        const long long share = (static_cast<long long>(sm_slots) * host_units + host_units + hbm_units - 1) /
                                (static_cast<long long>(host_units) + hbm_units);
        cap = std::max(cap, static_cast<int>(share));
    }
    cap = std::max(1, std::min(cap, sm_slots - (hbm_units > 0 ? 1 : 0)));
    if (host_units > 0 && hbm_units > 0 && !(t && (t->host_ctas > 0 || t->no_wave_align))) {
        // keep the HBM side at the wave count the whole operation would have on all slots:
        // host CTAs come out of the slack only (when a unit is compute-bound, one more HBM
        // wave costs a whole unit time, more than the host side saves)
        const int w0 = ceil_div(host_units + hbm_units, sm_slots);
        const int slack = sm_slots - ceil_div(hbm_units, w0);
        cap = std::max(1, std::min(cap, slack));
    }
    const bool align = !(t && t->no_wave_align);
    if (host_units > 0) {
        const int waves = ceil_div(host_units, cap);
        // whole waves: no partial tail wave
        s.n_host_ctas = align ? ceil_div(host_units, waves) : std::min(cap, host_units);
    }
    int hbm_slots = sm_slots - s.n_host_ctas;
    if (t && t->hbm_ctas > 0) hbm_slots = std::min(hbm_slots, t->hbm_ctas);
    hbm_slots = std::max(1, hbm_slots);
    if (hbm_units > 0) {
        const int waves = ceil_div(hbm_units, hbm_slots);
        s.n_hbm_ctas = align ? ceil_div(hbm_units, waves) : std::min(hbm_slots, hbm_units);
    }
    int hw = (t && t->window > 0) ? t->window : default_host_window;
    int bw = (t && t->hbm_window > 0) ? t->hbm_window : default_hbm_window;
    s.host_window = std::max(1, std::min(hw, max_window));
    s.hbm_window = std::max(1, std::min(bw, max_window));
    return s;
}

// ------------------------------------------------------------------------------------
// placement
// ------------------------------------------------------------------------------------

// Row-major A rows [rows][lda] (16-byte units of 8 bf16) -> the tile rows of one tier,
// tier-local tile rows l0, l0 + 1, ... (units / (KG * 64) of them). Tiles of 64 rows are
// stored [K_pad/8][64][8]: unit (l, kg, r) at l*KG*64 + kg*64 + r. Tiles of 128 rows
// (pairs) hold tile rows 2b and 2b + 1 of 64 as [K_pad/8][128][8]: unit (l, kg, r) at
// (l - l%2)*KG*64 + kg*128 + (l%2)*64 + r. Rows past `rows` and k-groups past K/8 are zero.
// With src_b set, packed row j comes from row j/2 of src (j even) or of src_b (j odd): the
// gate/up interleave of a SwiGLU weight.
__global__ void pack_matrix_kernel(const uint4* __restrict__ src, const uint4* __restrict__ src_b, long long lda16,
                                   long long rows, int K16, int KG, uint4* __restrict__ tier, long long l0,
                                   int pairs, long long units) {
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < units;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long per_tile = static_cast<long long>(KG) * kTileM;
        const long long t = idx / per_tile;
        const int rem = static_cast<int>(idx - t * per_tile);
        const int kg = rem / kTileM;
        const int r = rem - kg * kTileM;
        const long long row = t * kTileM + r;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row < rows && kg < K16) {
            v = src_b ? ((row & 1) ? src_b : src)[(row >> 1) * lda16 + kg] : src[row * lda16 + kg];
        }
        const long long l = l0 + t;
        const long long half = pairs ? (l & 1) : 0;
        const int rows_kg = pairs ? 2 * kTileM : kTileM;  // rows of one k-group of the tile
        tier[(l - half) * per_tile + static_cast<long long>(kg) * rows_kg + half * kTileM + r] = v;
    }
}

// K or V rows of `n_heads` (request, kv head) slabs, [n_heads][L][D] -> the chunked slab
// layout of the placement: per slab, chunks of 64 tokens [K 64 x D][V 64 x D] (last chunk
// zero-padded), and inside a token row the 16-byte piece c stored at c ^ (token & 7) so that
// ldmatrix reads of 8 consecutive tokens hit 8 different bank groups. `is_v` selects the
// half of each chunk.
__global__ void pack_kv_kernel(const uint4* __restrict__ src, long long n_heads, int L, int D16, int is_v,
                               long long slab16, uint4* __restrict__ dst) {
    const long long per_head = static_cast<long long>(L) * D16;
    const long long n_units = n_heads * per_head;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < n_units;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long head = idx / per_head;
        const long long rem = idx - head * per_head;
        const int j = static_cast<int>(rem / D16);
        const int c = static_cast<int>(rem - static_cast<long long>(j) * D16);
        const long long chunk = j >> 6;
        const long long off = head * slab16 + chunk * (2ll * 64 * D16) + (is_v ? 64ll * D16 : 0ll) +
                              static_cast<long long>(j & 63) * D16 + (c ^ (j & 7));
        dst[off] = src[idx];
    }
}

static void free_parts(dak_placement* p) {
    if (!p) return;
    host_free(p->host_ptr);
    dev_free(p->hbm_ptr);
    p->host_ptr = p->host_dev = p->hbm_ptr = nullptr;
}

static dak_status alloc_tiers(dak_placement* p) {
    if (p->host_bytes > 0) {
        if (host_alloc_mapped(&p->host_ptr, static_cast<size_t>(p->host_bytes)) != cudaSuccess) {
            cudaGetLastError();
            p->host_ptr = nullptr;
            return DAK_ERR_HOST_ALLOC;
        }
        if (cudaHostGetDevicePointer(&p->host_dev, p->host_ptr, 0) != cudaSuccess) {
            cudaGetLastError();
            return DAK_ERR_HOST_ALLOC;
        }
    }
    if (p->hbm_bytes > 0) {
        if (dev_alloc(&p->hbm_ptr, static_cast<size_t>(p->hbm_bytes)) != cudaSuccess) {
            cudaGetLastError();
            p->hbm_ptr = nullptr;
            return DAK_ERR_DEVICE_ALLOC;
        }
    }
    return DAK_OK;
}

static int pack_grid(long long units) {
    long long g = (units + 255) / 256;
    return static_cast<int>(std::max(1ll, std::min(g, 4096ll)));
}

}  // namespace dak

using namespace dak;

extern "C" const char* dak_status_string(int s) {
    switch (s) {
        case DAK_OK: return "ok";
        case DAK_ERR_INVALID: return "invalid argument";
        case DAK_ERR_ALIGN: return "misaligned pointer or size";
        case DAK_ERR_HOST_ALLOC: return "pinned host allocation failed";
        case DAK_ERR_DEVICE_ALLOC: return "device allocation failed";
        case DAK_ERR_CUDA: return "CUDA error";
        case DAK_ERR_TIMEOUT: return "kernel wait timed out";
        case DAK_ERR_UNSUPPORTED: return "unsupported shape";
        case DAK_ERR_BOUNDS: return "kernel index check failed";
        default: return "unknown status";
    }
}

// glu: A_src holds [2f][K] (f gate rows, then f up rows) with M = 2f; the placement stores
// them interleaved (row 2j = gate j, row 2j + 1 = up j).
static dak_status place_matrix(const void* A_src, int src_on_device, int64_t M, int64_t K, int64_t lda, int tile_m,
                               int n_host_tiles, bool glu, dak_placement** out) {
    if (!out) return DAK_ERR_INVALID;
    *out = nullptr;
    if (M < 0 || K <= 0 || lda < K || (M > 0 && !A_src)) return DAK_ERR_INVALID;
    if (glu && (M % kTileM)) return DAK_ERR_INVALID;  // whole tiles of 32 gate + 32 up rows
    if (tile_m != kTileM && tile_m != 2 * kTileM) return DAK_ERR_UNSUPPORTED;
    if ((K % 8) || (lda % 8) || (reinterpret_cast<uintptr_t>(A_src) & 15)) return DAK_ERR_ALIGN;
    if (K > (1 << 24) || M > (1ll << 31)) return DAK_ERR_INVALID;
    // internally every tier is counted in tile rows of 64: a 128-row tile is two of them (the
    // second all zero rows when the matrix ends in its first half)
    const int per = tile_m / kTileM;
    const int tiles = static_cast<int>((M + tile_m - 1) / tile_m);
    if (n_host_tiles < 0 || n_host_tiles > tiles) return DAK_ERR_INVALID;
    const int T = tiles * per;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DAK_ERR_CUDA;

    dak_placement* p = new dak_placement();
    std::memset(p, 0, sizeof(*p));
    p->kind = 0;
    p->device = dev;
    p->glu = glu ? 1 : 0;
    p->M = M;
    p->K = K;
    p->K_pad = (K + 15) / 16 * 16;
    p->tile_m = tile_m;
    p->T = T;
    p->h = n_host_tiles * per;
    p->tile_bytes = static_cast<int64_t>(kTileM) * p->K_pad * 2;
    p->host_bytes = p->tile_bytes * p->h;
    p->hbm_bytes = p->tile_bytes * (T - p->h);
    dak_status st = alloc_tiers(p);
    if (st != DAK_OK) {
        free_parts(p);
        delete p;
        return st;
    }

    // pack in batches of tile rows through a device staging buffer when the source is host memory
    const int KG = static_cast<int>(p->K_pad / 8);
    const int K16 = static_cast<int>(K / 8);
    const long long lda16 = lda / 8;
    const int batch_tiles = std::max(1, static_cast<int>((256ll << 20) / std::max<int64_t>(1, kTileM * lda * 2)));
    void* tmp = nullptr;
    cudaError_t e = cudaSuccess;
    if (!src_on_device && M > 0) {
        e = dev_alloc(&tmp, static_cast<size_t>(batch_tiles) * kTileM * lda * 2);
        if (e != cudaSuccess) {
            cudaGetLastError();
            free_parts(p);
            delete p;
            return DAK_ERR_DEVICE_ALLOC;
        }
    }
    const int64_t f = M / 2;
    for (int t0 = 0; t0 < T && e == cudaSuccess; t0 += batch_tiles) {
        const int nt = std::min(batch_tiles, T - t0);
        const long long row0 = static_cast<long long>(t0) * kTileM;
        // (0 for a batch holding only the zero second half of the last 128-row tile)
        const long long rows = std::max(0ll, std::min<long long>(static_cast<long long>(nt) * kTileM, M - row0));
        const uint8_t* a8 = static_cast<const uint8_t*>(A_src);
        const uint4* src;
        const uint4* src_b = nullptr;  // glu: the up rows (src: the gate rows)
        if (glu) {
            const long long g0 = row0 / 2, n_rows = rows / 2;
            if (src_on_device) {
                src = reinterpret_cast<const uint4*>(a8 + g0 * lda * 2);
                src_b = reinterpret_cast<const uint4*>(a8 + (f + g0) * lda * 2);
            } else {
                uint8_t* t8 = static_cast<uint8_t*>(tmp);
                e = cudaMemcpy(t8, a8 + g0 * lda * 2, static_cast<size_t>(n_rows * lda * 2), cudaMemcpyHostToDevice);
                if (e == cudaSuccess)
                    e = cudaMemcpy(t8 + n_rows * lda * 2, a8 + (f + g0) * lda * 2, static_cast<size_t>(n_rows * lda * 2),
                                   cudaMemcpyHostToDevice);
                src = reinterpret_cast<const uint4*>(t8);
                src_b = reinterpret_cast<const uint4*>(t8 + n_rows * lda * 2);
            }
        } else if (src_on_device) {
            src = reinterpret_cast<const uint4*>(a8 + row0 * lda * 2);
        } else {
            e = cudaMemcpy(tmp, a8 + row0 * lda * 2, static_cast<size_t>(rows * lda * 2), cudaMemcpyHostToDevice);
            src = reinterpret_cast<const uint4*>(tmp);
        }
        if (e != cudaSuccess) break;
        // destination: tile rows may straddle the tier boundary; pack each tier's part
        for (int tier = 0; tier < 2; ++tier) {
            const int lo = tier == 0 ? t0 : std::max(t0, p->h);
            const int hi = tier == 0 ? std::min(t0 + nt, p->h) : t0 + nt;
            if (hi <= lo) continue;
            uint8_t* base = static_cast<uint8_t*>(tier == 0 ? p->host_dev : p->hbm_ptr);
            const int first = tier == 0 ? 0 : p->h;  // first tile row stored in this tier
            const long long units = static_cast<long long>(hi - lo) * KG * kTileM;
            const long long src_row0 = static_cast<long long>(lo - t0) * kTileM;
            const long long src_rows = std::max(0ll, rows - src_row0);
            // glu: packed row j of this part reads row j/2 of the gate or up block
            const long long off = glu ? (src_row0 / 2) * lda16 : src_row0 * lda16;
            pack_matrix_kernel<<<pack_grid(units), 256>>>(src + off, src_b ? src_b + off : nullptr, lda16, src_rows,
                                                          K16, KG, reinterpret_cast<uint4*>(base), lo - first,
                                                          per == 2 ? 1 : 0, units);
            e = cudaGetLastError();
        }
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
    }
    dev_free(tmp);
    if (e != cudaSuccess) {
        cudaGetLastError();
        free_parts(p);
        delete p;
        return DAK_ERR_CUDA;
    }
    *out = p;
    return DAK_OK;
}

extern "C" dak_status dak_place_matrix(const void* A_src, int src_on_device, int64_t M, int64_t K, int64_t lda,
                                       int tile_m, int n_host_tiles, dak_placement** out) {
    return place_matrix(A_src, src_on_device, M, K, lda, tile_m, n_host_tiles, false, out);
}

extern "C" dak_status dak_place_matrix_glu(const void* A_src, int src_on_device, int64_t f, int64_t K, int64_t lda,
                                           int tile_m, int n_host_tiles, dak_placement** out) {
    if (f <= 0) {
        if (out) *out = nullptr;
        return DAK_ERR_INVALID;
    }
    return place_matrix(A_src, src_on_device, 2 * f, K, lda, tile_m, n_host_tiles, true, out);
}

extern "C" dak_status dak_place_kv_heads(const void* K_src, const void* V_src, int src_on_device, int B, int H_kv,
                                         int L, int D, int n_host_heads, dak_placement** out) {
    if (!out) return DAK_ERR_INVALID;
    *out = nullptr;
    if (B <= 0 || H_kv <= 0 || L <= 0 || !K_src || !V_src) return DAK_ERR_INVALID;
    if (static_cast<long long>(B) * H_kv > (1ll << 30)) return DAK_ERR_INVALID;
    if (D != 64 && D != 128) return DAK_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(K_src) & 15) || (reinterpret_cast<uintptr_t>(V_src) & 15)) return DAK_ERR_ALIGN;
    const int S = B * H_kv;  // (request, kv head) slabs, request-major
    if (n_host_heads < 0 || n_host_heads > S) return DAK_ERR_INVALID;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DAK_ERR_CUDA;

    dak_placement* p = new dak_placement();
    std::memset(p, 0, sizeof(*p));
    p->kind = 1;
    p->device = dev;
    p->B = B;
    p->H_kv = H_kv;
    p->L = L;
    p->D = D;
    p->h_s = n_host_heads;
    const int64_t n_chunks = (L + 63) / 64;
    p->head_bytes = n_chunks * 2 * 64 * D * 2;  // one (request, kv head) slab: K and V chunks
    const int64_t src_slab_bytes = static_cast<int64_t>(L) * D * 2;  // K (or V) of one slab in the source
    p->host_bytes = p->head_bytes * p->h_s;
    p->hbm_bytes = p->head_bytes * (S - p->h_s);
    dak_status st = alloc_tiers(p);
    if (st != DAK_OK) {
        free_parts(p);
        delete p;
        return st;
    }
    // zero both tiers first: the padding rows of every last chunk must hold finite values
    cudaError_t e = cudaSuccess;
    if (p->host_bytes) std::memset(p->host_ptr, 0, static_cast<size_t>(p->host_bytes));
    if (p->hbm_bytes) e = cudaMemset(p->hbm_ptr, 0, static_cast<size_t>(p->hbm_bytes));
    const int D16 = D / 8;
    const int batch = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(S, (256ll << 20) / src_slab_bytes)));
    void* tmp = nullptr;
    if (!src_on_device && e == cudaSuccess) {
        e = dev_alloc(&tmp, static_cast<size_t>(batch) * src_slab_bytes);
        if (e != cudaSuccess) {
            cudaGetLastError();
            free_parts(p);
            delete p;
            return DAK_ERR_DEVICE_ALLOC;
        }
    }
    for (int kv = 0; kv < 2 && e == cudaSuccess; ++kv) {
        const uint8_t* srcb = static_cast<const uint8_t*>(kv == 0 ? K_src : V_src);
        int ns = 0;
        for (int s0 = 0; s0 < S && e == cudaSuccess; s0 += ns) {
            // a batch of slabs (the source holds each slab contiguously), kept within one tier
            ns = std::min(batch, S - s0);
            if (s0 < p->h_s) ns = std::min(ns, p->h_s - s0);
            const uint4* src;
            if (src_on_device) {
                src = reinterpret_cast<const uint4*>(srcb + static_cast<long long>(s0) * src_slab_bytes);
            } else {
                e = cudaMemcpy(tmp, srcb + static_cast<long long>(s0) * src_slab_bytes,
                               static_cast<size_t>(ns) * src_slab_bytes, cudaMemcpyHostToDevice);
                src = reinterpret_cast<const uint4*>(tmp);
            }
            if (e != cudaSuccess) break;
            const bool host = s0 < p->h_s;
            const int ls = host ? s0 : s0 - p->h_s;
            uint8_t* tier = static_cast<uint8_t*>(host ? p->host_dev : p->hbm_ptr);
            uint8_t* dstb = tier + static_cast<long long>(ls) * p->head_bytes;
            const long long n_heads = ns;
            const long long units = n_heads * L * D16;
            pack_kv_kernel<<<pack_grid(units), 256>>>(src, n_heads, L, D16, kv, p->head_bytes / 16,
                                                      reinterpret_cast<uint4*>(dstb));
            e = cudaGetLastError();
            if (e == cudaSuccess) e = cudaDeviceSynchronize();
        }
    }
    dev_free(tmp);
    if (e != cudaSuccess) {
        cudaGetLastError();
        free_parts(p);
        delete p;
        return DAK_ERR_CUDA;
    }
    *out = p;
    return DAK_OK;
}

extern "C" dak_status dak_place_kv(const void* K_src, const void* V_src, int src_on_device, int B, int H_kv, int L,
                                   int D, int n_host_requests, dak_placement** out) {
    // whole requests: their H_kv slabs each (an out-of-range count stays out of range)
    const bool ok = B > 0 && H_kv > 0 && static_cast<long long>(B) * H_kv <= (1ll << 30) && n_host_requests >= 0 &&
                    n_host_requests <= B;
    return dak_place_kv_heads(K_src, V_src, src_on_device, B, H_kv, L, D, ok ? n_host_requests * H_kv : -1, out);
}

extern "C" dak_status dak_inject_fault(int kind, int skip, int count) {
    if (kind < 1 || kind >= kFaultKinds || skip < 0 || count < -1) return DAK_ERR_INVALID;
    load_fault_env();
    std::lock_guard<std::mutex> lock(g_fault_mu);
    g_fault_skip[kind] = skip;
    g_fault_count[kind] = count;
    return DAK_OK;
}

extern "C" int dak_fault_pending(int kind) {
    if (kind < 1 || kind >= kFaultKinds) return 0;
    load_fault_env();
    std::lock_guard<std::mutex> lock(g_fault_mu);
    return g_fault_count[kind];
}

extern "C" dak_status dak_alloc_counts(int64_t* host_live, int64_t* device_live) {
    if (host_live) *host_live = g_live_host.load();
    if (device_live) *device_live = g_live_dev.load();
    return DAK_OK;
}

extern "C" dak_status dak_free(dak_placement* p) {
    if (!p) return DAK_OK;
    free_parts(p);
    delete p;
    return DAK_OK;
}

extern "C" dak_status dak_placement_info(const dak_placement* p, int64_t* host_bytes, int64_t* hbm_bytes,
                                         int64_t* units, int64_t* host_units) {
    if (!p) return DAK_ERR_INVALID;
    if (host_bytes) *host_bytes = p->host_bytes;
    if (hbm_bytes) *hbm_bytes = p->hbm_bytes;
    const int per = (p->kind == 0 && p->tile_m > kTileM) ? p->tile_m / kTileM : 1;  // tiles, not 64-row rows
    if (units) *units = p->kind == 0 ? p->T / per : static_cast<int64_t>(p->B) * p->H_kv;
    if (host_units) *host_units = p->kind == 0 ? p->h / per : p->h_s;
    return DAK_OK;
}

extern "C" dak_status dak_last_error(void* stream, uint64_t* info) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return DAK_ERR_CUDA;
    DevStatus* st = status_ptr();
    if (!st) return DAK_ERR_CUDA;
    DevStatus h{};
    if (cudaMemcpy(&h, st, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return DAK_ERR_CUDA;
    if (h.code) {
        const DevStatus zero{};
        cudaMemcpy(st, &zero, sizeof(zero), cudaMemcpyHostToDevice);
        reset_split_counters();  // a GEMM that gave up may have counted only some pieces
    }
    if (info) *info = h.info;
    return static_cast<dak_status>(h.code);
}

extern "C" int dak_sm_count(void) { return device_sm_count(); }

// ------------------------------------------------------------------------------------
// tier read-stream probes (Fig. 7 experiments)
// ------------------------------------------------------------------------------------
namespace dak {

struct ProbeArgs {
    const uint8_t* buf[2];  // [0] host mapping, [1] HBM
    long long bytes[2];
    int ctas[2];
    int window[2];
    int chunk;
    int method;        // 0 bulk into smem, 1 ld.global.nc.v4, 2 tensor-map 2-D copy
    int verify;        // sum the words read
    unsigned long long* sums;     // per CTA
    unsigned long long* t_start;  // per CTA, globaltimer ns
    unsigned long long* t_end;
    DevStatus* st;
};

constexpr int kProbeThreads = 256;

__global__ void __launch_bounds__(kProbeThreads) probe_kernel(const ProbeArgs a, const __grid_constant__ CUtensorMap map) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint64_t full[16];
    __shared__ int abort_flag;
    volatile int* abort = &abort_flag;
    const int tier = blockIdx.x < a.ctas[0] ? 0 : 1;
    const int cta = tier == 0 ? blockIdx.x : blockIdx.x - a.ctas[0];
    const int nctas = a.ctas[tier];
    const int W = a.window[tier];
    const long long nchunks = a.bytes[tier] / a.chunk;
    const uint8_t* buf = a.buf[tier];
    unsigned long long sum = 0;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < W; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    const unsigned long long t0 = globaltimer();
    if (a.method == 1) {
        // every thread streams 16-byte non-coherent loads, `W` in flight
        const long long n16 = a.bytes[tier] / 16;
        const long long stride = static_cast<long long>(nctas) * kProbeThreads;
        for (long long base = static_cast<long long>(cta) * kProbeThreads + threadIdx.x; base < n16;
             base += stride * W) {
            uint4 v[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const long long idx = base + u * stride;
                if (u < W && idx < n16) v[u] = ld_nc_v4(buf + idx * 16);
            }
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const long long idx = base + u * stride;
                if (u < W && idx < n16) sum += static_cast<unsigned long long>(v[u].x) + v[u].y + v[u].z + v[u].w;
            }
        }
    } else {
        long long i = 0;
        for (long long c = cta; c < nchunks; c += nctas, ++i) {
            const int s = static_cast<int>(i % W);
            if (threadIdx.x == 0) {
                if (i >= W) {
                    // slot reuse: the consumer side below waited for it already
                }
                mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(a.chunk));
                if (a.method == 0) {
                    bulk_g2s(smem + static_cast<size_t>(s) * a.chunk, buf + c * a.chunk, static_cast<uint32_t>(a.chunk),
                             &full[s], policy_evict_first());
                } else {
                    // view: rows of 512 bytes (256 bf16); one box = chunk / 512 rows
                    const int rows = a.chunk / 512;
                    tma_load_2d(smem + static_cast<size_t>(s) * a.chunk, &map, 0, static_cast<int>(c * rows),
                                &full[s]);
                }
            }
            // keep W chunks in flight: wait for the chunk issued W-1 iterations ago
            if (i >= W - 1) {
                const long long j = i - (W - 1);
                const int sj = static_cast<int>(j % W);
                if (!mbar_wait(&full[sj], static_cast<uint32_t>((j / W) & 1), abort, a.st, DAK_ERR_TIMEOUT, 100)) break;
                if (a.verify) {
                    const uint32_t* w32 = reinterpret_cast<const uint32_t*>(smem + static_cast<size_t>(sj) * a.chunk);
                    for (int k = threadIdx.x; k < a.chunk / 4; k += kProbeThreads) sum += w32[k];
                }
                __syncthreads();  // slot sj may be refilled next iteration
            }
        }
        // drain the last W-1 chunks (bounded waits that ignore the abort flag)
        const long long issued = i;
        volatile int drain_flag = 0;
        for (long long j = issued > W - 1 ? issued - (W - 1) : 0; j < issued; ++j) {
            const int sj = static_cast<int>(j % W);
            if (!mbar_wait(&full[sj], static_cast<uint32_t>((j / W) & 1), &drain_flag, a.st, DAK_ERR_TIMEOUT, 101)) break;
            if (a.verify) {
                const uint32_t* w32 = reinterpret_cast<const uint32_t*>(smem + static_cast<size_t>(sj) * a.chunk);
                for (int k = threadIdx.x; k < a.chunk / 4; k += kProbeThreads) sum += w32[k];
            }
        }
    }
    // block reduction of the checksum
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    __shared__ unsigned long long red[kProbeThreads / 32];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sum;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long s = 0;
        for (int k = 0; k < kProbeThreads / 32; ++k) s += red[k];
        a.sums[blockIdx.x] = s;
        a.t_start[blockIdx.x] = t0;
        a.t_end[blockIdx.x] = globaltimer();
    }
}

__global__ void fill_pattern_kernel(uint32_t* p, long long n, long long offset) {
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        p[i] = static_cast<uint32_t>((offset + i) * 2654435761ull);
    }
}

static unsigned long long pattern_sum(long long n_words) {
    unsigned long long s = 0;
    for (long long i = 0; i < n_words; ++i) s += static_cast<uint32_t>(i * 2654435761ull);
    return s;
}

using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;
static EncodeTiledFn probe_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
        }
    });
    return fn;
}

struct ProbeBuffers {
    void* host = nullptr;
    void* host_dev = nullptr;
    void* hbm = nullptr;
    long long host_bytes = 0, hbm_bytes = 0;
    ~ProbeBuffers() {
        host_free(host);
        dev_free(hbm);
    }
};

static dak_status probe_alloc(ProbeBuffers& b, long long host_bytes, long long hbm_bytes) {
    if (host_bytes > 0) {
        if (host_alloc_mapped(&b.host, host_bytes) != cudaSuccess) {
            cudaGetLastError();
            b.host = nullptr;
            return DAK_ERR_HOST_ALLOC;
        }
        cudaHostGetDevicePointer(&b.host_dev, b.host, 0);
        b.host_bytes = host_bytes;
        uint32_t* w = static_cast<uint32_t*>(b.host);
        const long long n = host_bytes / 4;
        for (long long i = 0; i < n; ++i) w[i] = static_cast<uint32_t>(i * 2654435761ull);
    }
    if (hbm_bytes > 0) {
        if (dev_alloc(&b.hbm, hbm_bytes) != cudaSuccess) {
            cudaGetLastError();
            b.hbm = nullptr;
            return DAK_ERR_DEVICE_ALLOC;
        }
        b.hbm_bytes = hbm_bytes;
        fill_pattern_kernel<<<1024, 256>>>(static_cast<uint32_t*>(b.hbm), hbm_bytes / 4, 0);
        if (cudaDeviceSynchronize() != cudaSuccess) return DAK_ERR_CUDA;
    }
    return DAK_OK;
}

// Run the probe kernel `iters` times; per tier keep the best bandwidth (bytes / busy span).
static dak_status probe_run(ProbeBuffers& b, int method, int host_ctas, int host_window, int hbm_ctas, int hbm_window,
                            int chunk, int iters, double* gbps_host, double* gbps_hbm, int* ok) {
    ProbeArgs a{};
    a.buf[0] = static_cast<const uint8_t*>(b.host_dev);
    a.buf[1] = static_cast<const uint8_t*>(b.hbm);
    a.bytes[0] = host_ctas > 0 ? (b.host_bytes / chunk) * chunk : 0;
    a.bytes[1] = hbm_ctas > 0 ? (b.hbm_bytes / chunk) * chunk : 0;
    a.ctas[0] = host_ctas;
    a.ctas[1] = hbm_ctas;
    a.window[0] = std::max(1, std::min(host_window, 16));
    a.window[1] = std::max(1, std::min(hbm_window, 16));
    a.chunk = chunk;
    a.method = method;
    a.st = status_ptr();
    if (!a.st) return DAK_ERR_CUDA;
    const int grid = host_ctas + hbm_ctas;
    if (grid <= 0) return DAK_ERR_INVALID;
    std::vector<unsigned long long> h_sums(grid), h_t0(grid), h_t1(grid);
    unsigned long long* d = nullptr;
    if (dev_alloc(reinterpret_cast<void**>(&d), sizeof(unsigned long long) * 3 * grid) != cudaSuccess)
        return DAK_ERR_DEVICE_ALLOC;
    a.sums = d;
    a.t_start = d + grid;
    a.t_end = d + 2 * grid;
    alignas(64) CUtensorMap map;
    std::memset(&map, 0, sizeof(map));
    if (method == 2) {
        EncodeTiledFn enc = probe_encode_fn();
        const uint8_t* tbuf = host_ctas > 0 ? a.buf[0] : a.buf[1];
        const long long tbytes = host_ctas > 0 ? a.bytes[0] : a.bytes[1];
        if (!enc || (host_ctas > 0 && hbm_ctas > 0) || chunk % 512 || chunk / 512 > 256) {
            dev_free(d);
            return DAK_ERR_UNSUPPORTED;
        }
        cuuint64_t dims[2] = {256, static_cast<cuuint64_t>(tbytes / 512)};
        cuuint64_t strides[1] = {512};
        cuuint32_t box[2] = {256, static_cast<cuuint32_t>(chunk / 512)};
        cuuint32_t estr[2] = {1, 1};
        if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint8_t*>(tbuf), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
            dev_free(d);
            return DAK_ERR_UNSUPPORTED;  // the tensor map does not encode over this memory
        }
    }
    const int smem = method == 1 ? 0 : std::max(a.window[0], a.window[1]) * chunk;
    if (smem > 220 * 1024) {
        dev_free(d);
        return DAK_ERR_INVALID;
    }
    cudaFuncSetAttribute(probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    double best[2] = {0, 0};
    int data_ok = 1;
    for (int it = 0; it < iters + 1; ++it) {
        a.verify = (it == 0) ? 1 : 0;
        probe_kernel<<<grid, kProbeThreads, smem>>>(a, map);
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess) {
            dev_free(d);
            return DAK_ERR_CUDA;
        }
        cudaMemcpy(h_sums.data(), a.sums, sizeof(unsigned long long) * grid, cudaMemcpyDeviceToHost);
        cudaMemcpy(h_t0.data(), a.t_start, sizeof(unsigned long long) * grid, cudaMemcpyDeviceToHost);
        cudaMemcpy(h_t1.data(), a.t_end, sizeof(unsigned long long) * grid, cudaMemcpyDeviceToHost);
        for (int tier = 0; tier < 2; ++tier) {
            const int lo = tier == 0 ? 0 : host_ctas, hi = tier == 0 ? host_ctas : grid;
            if (hi <= lo || a.bytes[tier] == 0) continue;
            unsigned long long mn = ~0ull, mx = 0, s = 0;
            for (int k = lo; k < hi; ++k) {
                mn = std::min(mn, h_t0[k]);
                mx = std::max(mx, h_t1[k]);
                s += h_sums[k];
            }
            if (it == 0) {
                if (s != pattern_sum(a.bytes[tier] / 4)) data_ok = 0;
                continue;
            }
            const double gbps = mx > mn ? static_cast<double>(a.bytes[tier]) / static_cast<double>(mx - mn) : 0.0;
            best[tier] = std::max(best[tier], gbps);
        }
    }
    dev_free(d);
    if (gbps_host) *gbps_host = best[0];
    if (gbps_hbm) *gbps_hbm = best[1];
    if (ok) *ok = data_ok;
    DevStatus h{};
    cudaMemcpy(&h, a.st, sizeof(h), cudaMemcpyDeviceToHost);
    if (h.code) {
        const DevStatus zero{};
        cudaMemcpy(a.st, &zero, sizeof(zero), cudaMemcpyHostToDevice);
        return static_cast<dak_status>(h.code);
    }
    return DAK_OK;
}

}  // namespace dak

extern "C" dak_status dak_probe_read_bw(int tier, int64_t bytes, int method, int ctas, int window, int chunk_bytes,
                                        int iters, double* gbps_out, int* data_ok_out) {
    if ((tier != 0 && tier != 1) || bytes <= 0 || ctas <= 0 || window <= 0 || chunk_bytes < 16 ||
        (chunk_bytes % 16) || method < 0 || method > 2 || iters <= 0)
        return DAK_ERR_INVALID;
    dak::ProbeBuffers b;
    dak_status st = dak::probe_alloc(b, tier == 0 ? bytes : 0, tier == 1 ? bytes : 0);
    if (st != DAK_OK) return st;
    double h = 0, g = 0;
    st = dak::probe_run(b, method, tier == 0 ? ctas : 0, window, tier == 1 ? ctas : 0, window, chunk_bytes, iters, &h,
                        &g, data_ok_out);
    if (gbps_out) *gbps_out = tier == 0 ? h : g;
    return st;
}

extern "C" dak_status dak_probe_concurrent(int64_t host_bytes, int64_t hbm_bytes, int host_ctas, int host_window,
                                           int hbm_ctas, int hbm_window, int chunk_bytes, int iters, double* host_gbps,
                                           double* hbm_gbps) {
    if (host_bytes <= 0 || hbm_bytes <= 0 || host_ctas < 0 || hbm_ctas < 0 || chunk_bytes < 16 ||
        (chunk_bytes % 16) || iters <= 0)
        return DAK_ERR_INVALID;
    dak::ProbeBuffers b;
    dak_status st = dak::probe_alloc(b, host_bytes, hbm_bytes);
    if (st != DAK_OK) return st;
    int ok = 1;
    return dak::probe_run(b, 0, host_ctas, host_window, hbm_ctas, hbm_window, chunk_bytes, iters, host_gbps, hbm_gbps,
                          &ok);
}

// One CTA waits on an mbarrier that nothing arrives at: the bounded wait must run out,
// record DAK_ERR_TIMEOUT and let the kernel return normally.
__global__ void selftest_wait_kernel(DevStatus* st) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    mbar_wait(&bar, 0, &abort_flag, st, DAK_ERR_TIMEOUT, 0x5E1Fu);
}

extern "C" dak_status dak_selftest_wait(void* stream) {
    DevStatus* st = status_ptr();
    if (!st) return DAK_ERR_CUDA;
    selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(st);
    return cuda_status(cudaGetLastError());
}

// One thread waits for a handoff count that nothing raises: the pacing wait gives up after
// its bound, counts itself in link_timeouts and the kernel returns normally.
__global__ void selftest_link_kernel(const unsigned* never, DevStatus* st) { link_wait(never, 1u, st); }

extern "C" dak_status dak_selftest_link(void* stream) {
    DevStatus* st = status_ptr();
    if (!st) return DAK_ERR_CUDA;
    void* zero = nullptr;  // a count that stays at zero
    if (dev_alloc(&zero, sizeof(unsigned)) != cudaSuccess) return DAK_ERR_DEVICE_ALLOC;
    cudaError_t e = cudaMemsetAsync(zero, 0, sizeof(unsigned), static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) {
        selftest_link_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<const unsigned*>(zero), st);
        e = cudaGetLastError();
    }
    const cudaError_t s = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    dev_free(zero);
    return cuda_status(e != cudaSuccess ? e : s);
}

extern "C" dak_status dak_link_timeouts(void* stream, uint32_t* count) {
    if (!count) return DAK_ERR_INVALID;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return DAK_ERR_CUDA;
    DevStatus* st = status_ptr();
    if (!st) return DAK_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpy(&v, &st->link_timeouts, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return DAK_ERR_CUDA;
    if (v) {
        const unsigned z = 0;
        if (cudaMemcpy(&st->link_timeouts, &z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess) return DAK_ERR_CUDA;
    }
    *count = v;
    return DAK_OK;
}

// Append one token's key and value per (request, kv head) to a placed cache: block (b, g)
// writes k_new[b][g] and v_new[b][g] into the slab of (b, g), in whichever tier holds it, at
// row positions[b] of its chunk layout (16-byte piece c of token j stored at c ^ (j mod 8)).
// A position outside [0, L) is skipped and reported (DAK_ERR_BOUNDS, info = request).
__global__ void kv_append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                 const int* __restrict__ positions, uint8_t* host, uint8_t* hbm, long long head_bytes,
                                 int H_kv, int D16, int L, int h_s, DevStatus* st) {
    const int b = blockIdx.x, g = blockIdx.y;
    const int pos = positions[b];
    if (pos < 0 || pos >= L) {
        if (g == 0 && threadIdx.x == 0) report(st, DAK_ERR_BOUNDS, 0xA9900000ull | static_cast<unsigned>(b));
        return;
    }
    const long long slab = static_cast<long long>(b) * H_kv + g;
    uint4* base = reinterpret_cast<uint4*>(slab < h_s ? host + slab * head_bytes : hbm + (slab - h_s) * head_bytes);
    const long long row = static_cast<long long>(pos >> 6) * (2 * 64 * D16) + static_cast<long long>(pos & 63) * D16;
    for (int t = threadIdx.x; t < 2 * D16; t += blockDim.x) {
        const bool is_v = t >= D16;
        const int c = is_v ? t - D16 : t;
        const uint4 piece = (is_v ? v_new : k_new)[slab * D16 + c];
        base[row + (is_v ? 64 * D16 : 0) + (c ^ (pos & 7))] = piece;
    }
}

extern "C" dak_status dak_kv_append(const dak_placement* KV, const void* k_new, const void* v_new,
                                    const int* positions, void* stream) {
    if (!KV || KV->kind != 1 || !k_new || !v_new || !positions) return DAK_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(k_new) & 15) || (reinterpret_cast<uintptr_t>(v_new) & 15)) return DAK_ERR_ALIGN;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DAK_ERR_CUDA;
    if (dev != KV->device) return DAK_ERR_INVALID;
    DevStatus* st = status_ptr();
    if (!st) return DAK_ERR_CUDA;
    const int D16 = KV->D / 8;
    kv_append_kernel<<<dim3(static_cast<unsigned>(KV->B), static_cast<unsigned>(KV->H_kv)), 2 * D16, 0,
                       static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), positions,
        static_cast<uint8_t*>(KV->host_dev), static_cast<uint8_t*>(KV->hbm_ptr), KV->head_bytes, KV->H_kv, D16,
        KV->L, KV->h_s, st);
    return cuda_status(cudaGetLastError());
}

extern "C" dak_status dak_prefetch(const dak_placement* p, void* staging, void* stream) {
    if (!p) return DAK_ERR_INVALID;
    if (p->host_bytes == 0) return DAK_OK;
    if (!staging) return DAK_ERR_INVALID;
    // copy-engine copy addressed through the device-visible alias of the pinned buffer
    // (cudaMemcpyDefault): on GB300 this form held 209-211 GB/s where the host-pointer
    // form fell to 30-90 GB/s on freshly touched or very large pinned regions
    return dak::cuda_status(cudaMemcpyAsync(staging, p->host_dev, static_cast<size_t>(p->host_bytes),
                                            cudaMemcpyDefault, static_cast<cudaStream_t>(stream)));
}
