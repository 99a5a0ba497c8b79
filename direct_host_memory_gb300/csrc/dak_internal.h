// Library-internal declarations shared by the runtime, GEMM and attention translation units.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/dak.h"

struct dak_placement {
    int kind;    // 0 = matrix (GEMM weights), 1 = KV cache
    int device;  // device the placement was made on
    int glu;     // matrix: gate/up rows interleaved (row 2j gate j, row 2j+1 up j); dak_gemm applies SwiGLU
    // tier buffers: host part (pinned, device-mapped; host and device addresses) and HBM part
    void* host_ptr;
    void* host_dev;
    void* hbm_ptr;
    int64_t host_bytes;
    int64_t hbm_bytes;
    // matrix
    int64_t M, K, K_pad;
    int tile_m;
    int T;  // tile rows
    int h;  // tile rows on the host
    int64_t tile_bytes;
    // kv
    int B, H_kv, L, D;
    int h_s;                // (request, kv head) slabs on the host: the first h_s in request-major order
    int64_t head_bytes;     // one (request, kv head) slab: ceil(L/64) chunks of [K 64 x D][V 64 x D] bf16
};

namespace dak {

constexpr int kTileM = 64;

// Device status block: first failure code and where it happened.
struct DevStatus {
    int code;
    unsigned link_timeouts;  // host-link handoff waits that gave up (dak_link_timeouts)
    unsigned long long info;
};

// Device address of the status block of the current device (set up once per device).
DevStatus* status_ptr();
// Zero the per-tile-row counters of split GEMM tile rows (after a kernel gave up midway).
void reset_split_counters();

struct Sched {
    int n_host_ctas;  // CTAs [0, n_host_ctas) read the host tier
    int n_hbm_ctas;   // CTAs [n_host_ctas, n_host_ctas + n_hbm_ctas) read HBM
    int host_window;
    int hbm_window;
};

// Split a persistent grid between the two tiers: (1) enough host CTAs for the host
// units, capped by the congestion limit; (2) whole waves on each side, so that no
// tail wave runs with a few CTAs; (3) every other SM on the HBM side.
Sched schedule(int host_units, int hbm_units, int sm_slots, const dak_tuning* t, int default_host_ctas,
               int default_host_window, int default_hbm_window, int max_window);

int device_sm_count();
dak_status cuda_status(cudaError_t e);

// Identifier of the current CUDA context, unique for the process's lifetime (0 if none): a
// device address looked up with cudaGetSymbolAddress is kept together with it, so that the
// address is looked up again after the context was destroyed and made anew.
unsigned long long current_context_id();

// The library's allocations go through these wrappers, which count the live allocations
// (dak_alloc_counts) and take the host-side fault injection of dak_inject_fault: an injected
// failure returns cudaErrorMemoryAllocation without calling CUDA.
cudaError_t host_alloc_mapped(void** p, size_t bytes);  // cudaHostAlloc(Mapped | Portable)
void host_free(void* p);
cudaError_t dev_alloc(void** p, size_t bytes);
void dev_free(void* p);
// True when an injected failure of this kind (DAK_FAULT_*) is due now (consumes it).
bool fault_due(int kind);

// kernel launchers (defined in dak_gemm.cu / dak_attn.cu)
// ws / ws_bytes: the caller's split workspace (dak_gemm_ws), or null for the module's own
// A decode step's RMSNorm folded into the GEMMs around it (all members null = off).
// Producer (res_x): the launch adds its product to the fp32 residual x [N][M] in place and
// writes C = bf16(x * g) (bf16 [N][M]) and ss_out [T][N], the sums of x^2 over each tile
// row's 64 rows. Consumer (ss_in): the accumulators of hidden-state row n are multiplied by
// 1 / sqrt(sum_t ss_in[t][n] * inv_d + eps) (t < ss_tiles) before they are stored. N <= 128.
struct GemmFuse {
    float* res_x = nullptr;
    const void* res_g = nullptr;  // bf16 [M]
    float* ss_out = nullptr;
    const float* ss_in = nullptr;
    int ss_tiles = 0;
    float inv_d = 0.f, eps = 0.f;
};

// Host-link handoff of a sequence of launches on one stream, e.g. a decode step's kernels
// (link_wait / link_signal): ctr counts the host-tier producers of the sequence's launches
// that have issued their last load (zeroed when the sequence starts); this launch's host
// producers start once it reaches `after`. The launcher stores in *signals how many
// producers of this launch add to the count (0 for a launch without host tiles).
struct LinkHandoff {
    unsigned* ctr = nullptr;
    unsigned after = 0;
    int* signals = nullptr;
};
// Sequences of the public calls (dak_link_begin; a launch joins sequence t->link): the
// handoff a joining launch takes (false: the launch joins none), and the signals it adds.
constexpr int kLinkSlots = 8;
bool link_join(const dak_tuning* t, LinkHandoff* lk);
void link_commit(const dak_tuning* t, int signals);

// One operation of a chain of GEMMs run by one persistent launch (launch_gemm_chain):
// host_src is the host tier's device-visible address (or a prefetch staging copy);
// after_prev: B (and the fused inputs) come from earlier operations of the chain, so the
// operation's loads of B and its epilogue wait until every CTA has finished the previous one.
constexpr int kMaxChainOps = 8;
struct ChainOp {
    const dak_placement* A = nullptr;
    const void* host_src = nullptr;
    const void* B = nullptr;
    void* C = nullptr;
    int c_fp32 = 0;
    int after_prev = 0;
    GemmFuse fuse;
};
// ws: the chain's workspace (256-byte aligned, gemm_chain_workspace_bytes of it, zeroed before
// its first use; every completed launch leaves its counters at zero again).
dak_status launch_gemm_chain(const ChainOp* ops, int n, int N, const dak_tuning* t, void* ws, size_t ws_bytes,
                             cudaStream_t s);
size_t gemm_chain_workspace_bytes(const ChainOp* ops, int n, int N, const dak_tuning* t);

dak_status launch_gemm(const dak_placement* A, const void* host_src, const void* B, void* C, int N, int c_fp32,
                       const dak_tuning* t, cudaStream_t s, void* ws = nullptr, size_t ws_bytes = 0,
                       const GemmFuse* fuse = nullptr, const LinkHandoff* link = nullptr);
size_t gemm_workspace_bytes(const dak_placement* A, int N);
// o_fp32: O is fp32 [B][H_q][D] (dak_attn_f32) instead of bf16
dak_status launch_attn(const void* Q, const dak_placement* KV, const void* host_src, const int* seq_lens, int H_q,
                       float scale, void* O, void* ws, size_t ws_bytes, const dak_tuning* t, cudaStream_t s,
                       int o_fp32 = 0, const LinkHandoff* link = nullptr);

}  // namespace dak
