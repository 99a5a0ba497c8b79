// Decode attention for callers that cannot allocate device memory.
//
// dak_attn needs a device workspace for the partial results of the context splits, and
// the caller provides it. Some callers cannot allocate one on demand: an engine that has
// already reserved the device's memory for its own weight and KV-cache pools, code that
// has no handle on the allocator the rest of the process uses, or a latency-critical loop
// in which a cudaMalloc / cudaFree would synchronise the device. dak_attn_noalloc runs the
// same kernels with that workspace taken from a fixed array compiled into the library.
//
// The array lives in every device's memory from the moment the library's device code is
// loaded on that device until the process exits. All calls share it: calls that overlap
// on the GPU (different streams, no ordering between them) race on it. Nothing in it
// needs to start at zero: every call writes each partial result before reading it, so
// the previous call's leftovers are never read.
#include <mutex>

#include "dak_device.cuh"

namespace {

constexpr size_t kNoallocScratchBytes = DAK_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of the array on the current device. In host code the array's name is
// only a host-side handle, so the address is looked up once per device (with that device
// current) and kept, together with the identifier of the context it belongs to: after a
// cudaDeviceReset the context (and with it the array) is made anew at a new address, so a
// changed identifier means looking it up again.
void* noalloc_scratch_address() {
    static void* addr[64] = {nullptr};
    static unsigned long long ctx[64] = {0};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long id = dak::current_context_id();
    if (!addr[dev] || ctx[dev] != id) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        addr[dev] = p;
        ctx[dev] = dak::current_context_id();  // the lookup may have created the context
    }
    return addr[dev];
}

}  // namespace

extern "C" dak_status dak_attn_noalloc(const void* Q, const dak_placement* KV, const int* seq_lens, int H_q,
                                       float scale, void* O, const dak_tuning* tuning, void* stream) {
    if (!KV || KV->kind != 1 || H_q <= 0) return DAK_ERR_INVALID;
    const int n_split = (tuning && tuning->n_split > 0) ? tuning->n_split : dak_attn_default_split(KV);
    const size_t need = dak_attn_workspace_bytes(KV->B, H_q, KV->D, n_split);
    if (need > kNoallocScratchBytes) return DAK_ERR_INVALID;  // the fixed array is too small for this call
    void* ws = nullptr;
    if (need > 0) {
        ws = noalloc_scratch_address();
        if (!ws) return DAK_ERR_CUDA;
    }
    dak_tuning t{};
    if (tuning) t = *tuning;
    t.n_split = n_split;  // the launch uses the split the size check was made for
    return dak::launch_attn(Q, KV, KV->host_dev, seq_lens, H_q, scale, O, ws, need, &t,
                            static_cast<cudaStream_t>(stream));
}
